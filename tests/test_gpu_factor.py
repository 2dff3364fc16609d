"""GPU parity of the fixed top-K baseline, Fast-dLLM factor decoding and the
Theorem-1 certificate against the oracle (same fp32 inputs on both sides, so
selections must match bit for bit)."""
import numpy as np
import pytest
import torch

import oracle
import synth
from parity import oracle_stats

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dlm():
    import diffusion_decoding_token_gb300 as d
    d.lib()
    return d


def cuda(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _cases():
    rng = np.random.default_rng(12)
    out = []
    for blk in (1, 7, 32, 100, 256):
        for B in (1, 9):
            conf = (1 - rng.random((B, blk)) ** 2 * 0.7).astype(np.float32)
            conf[:, ::6] = np.float32(0.875)  # exact ties
            masked = (rng.random((B, blk)) < 0.75).astype(np.uint8)
            masked[0, :] = 1
            if B > 1:
                masked[1, :] = 0  # nothing masked
            out.append((conf, masked))
    return out


@pytest.mark.parametrize("case", range(10))
def test_topk_and_factor_random(dlm, case):
    conf, masked = _cases()[case]
    c64 = conf.astype(np.float64)
    for k in (0, 1, 3, 1000):
        gs, gn = dlm.select_topk(cuda(conf), cuda(masked), k)
        os_, on = oracle.select_topk(c64, masked, k)
        np.testing.assert_array_equal(gs.cpu().numpy(), os_)
        np.testing.assert_array_equal(gn.cpu().numpy(), on)
    for f in (0.01, 0.2, 1.0, 5.0):
        gs, gn = dlm.select_factor(cuda(conf), cuda(masked), f)
        os_, on = oracle.select_factor(c64, masked, f)
        np.testing.assert_array_equal(gs.cpu().numpy(), os_)
        np.testing.assert_array_equal(gn.cpu().numpy(), on)
        gc = dlm.parallel_certificate(cuda(conf), gs)
        oc = oracle.parallel_certificate(c64, os_)
        np.testing.assert_array_equal(gc.cpu().numpy(), oc)


@pytest.mark.parametrize("name", ["llada_step", "batched", "stress_graph"])
def test_rules_on_workload_confidences(dlm, name):
    w = synth.make(synth.scaled(synth.CONFIGS[name], vocab=4096), seed=41)
    o = oracle_stats(w)
    cfg = w.cfg
    c32 = o["conf"].astype(np.float32).reshape(cfg.batch, cfg.blk)
    c64 = c32.astype(np.float64)
    for rule in ("threshold", "factor", "topk"):
        if rule == "threshold":
            gs, _ = dlm.select_threshold(cuda(c32), cuda(w.masked), cfg.tau)
            os_, _ = oracle.select_threshold(c64, w.masked, cfg.tau)
        elif rule == "factor":
            gs, _ = dlm.select_factor(cuda(c32), cuda(w.masked), 1.0)
            os_, _ = oracle.select_factor(c64, w.masked, 1.0)
        else:
            gs, _ = dlm.select_topk(cuda(c32), cuda(w.masked), 4)
            os_, _ = oracle.select_topk(c64, w.masked, 4)
        np.testing.assert_array_equal(gs.cpu().numpy(), os_)
        gc = dlm.parallel_certificate(cuda(c32), gs)
        np.testing.assert_array_equal(gc.cpu().numpy(), oracle.parallel_certificate(c64, os_))
