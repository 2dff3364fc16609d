"""The bounded waits of the DAPD attention pass, made to run out on a healthy
GPU.

The bulk-copy attention kernel waits on an mbarrier for its own copies, with
a limit of about a second; when a wait runs out the kernel drains the copies
it issued (again with a bounded wait), sets DLM_DEV_TIMEOUT in the caller's
status word and stores none of that tile's sums.  A test hook of the library
(not declared in dlm.h) lowers the limit of the first wait of each CTA to a
few clock cycles of non-blocking probes, so the wait gives up while the copies
are still on their way: no fault and no hang, only the timeout path.  The
call must return, the status word must say so, and the next call on the same
stream with the normal limit must match the oracle.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import synth
from parity import DeviceWorkload, screen

pytestmark = pytest.mark.gpu


def _hook(dlm):
    L = dlm.lib()
    f = L.dlm_test_set_first_wait_limit
    f.restype = None
    f.argtypes = [ctypes.c_longlong]
    return f


@pytest.mark.parametrize("batch,blk", [(2, 64), (6, 200)])
def test_first_wait_runs_out_then_the_next_call_is_clean(batch, blk):
    import diffusion_decoding_token_gb300 as dlm
    set_limit = _hook(dlm)
    cfg = synth.scaled(synth.CONFIGS["stress_graph"], batch=batch, blk=blk, vocab=512,
                       seq_len=(blk + 64 + 7) // 8 * 8, block_start=64, rules=("dapd",))
    w, o = screen(cfg, seed=90 + blk, use_stored=False)
    dw = DeviceWorkload(w)
    conf = torch.from_numpy(np.asarray(o["conf"], np.float32).reshape(batch, blk)).cuda()
    args = (dw.attn, dw.masked, conf, cfg.tau_edge, cfg.bulk_conf, cfg.bulk_frac, 0, dw.block_start)
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        st = dlm.new_status()
        try:
            set_limit(8)                       # eight clock cycles: the first copy cannot have landed
            dlm.dapd_graph_mis(*args, status=st)
        finally:
            set_limit(-1)
        stream.synchronize()
        assert int(st.item()) & dlm.DEV_TIMEOUT
        st2 = dlm.new_status()
        gs, gn = dlm.dapd_graph_mis(*args, status=st2)
        stream.synchronize()
    assert int(st2.item()) == 0
    r = oracle.dapd(w.attn, w.masked, np.asarray(o["conf"], np.float32).astype(np.float64).reshape(batch, blk),
                    cfg.tau_edge, cfg.bulk_conf, cfg.bulk_frac, 0, dtype=synth.F16)
    np.testing.assert_array_equal(gs.cpu().numpy(), r["selected"])
    np.testing.assert_array_equal(gn.cpu().numpy(), r["n_selected"])
