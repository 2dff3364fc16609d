"""dlm_revocable_step against the oracle's step, bit for bit, over whole
multi-step runs from the same fp32 inputs: every state array, the outcomes
and the counts after every step.  Coarse confidence grids force ties in both
rankings; ragged blocks, blk = 1 and finished sequences are covered."""
import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu

KEYS = ("tok", "masked", "seed", "last_seed", "remasks", "last_tok", "flipflops")


def _run(B, blk, steps, seed, grid=None, V=4, **kw):
    import diffusion_decoding_token_gb300 as dlm
    rng = np.random.default_rng(seed)
    ost = oracle.revocable_init(B, blk)
    gst = dlm.revocable_state(B, blk, "cuda")
    for t in range(steps):
        am = rng.integers(0, V, (B, blk)).astype(np.int32)
        conf = (rng.random((B, blk)) ** 0.3).astype(np.float32)
        if grid:
            conf = (np.round(conf * grid) / grid).astype(np.float32)
        infl = (rng.random((B, blk)) * 2).astype(np.float32)
        drift = (rng.random((B, blk)) * 0.3).astype(np.float32)
        if grid:
            infl = (np.round(infl * grid) / grid).astype(np.float32)
            drift = np.zeros_like(drift)
        r = oracle.revocable_step(am, conf.astype(np.float64), ost, t, influence=infl.astype(np.float64),
                                  drift=drift.astype(np.float64), **kw)
        out, nd, nr = dlm.revocable_step(torch.from_numpy(am).cuda(), torch.from_numpy(conf).cuda(), gst, t,
                                         influence=torch.from_numpy(infl).cuda(),
                                         drift=torch.from_numpy(drift).cuda(), **kw)
        np.testing.assert_array_equal(out.cpu().numpy(), r["outcome"], err_msg=f"outcome, step {t}")
        np.testing.assert_array_equal(nd.cpu().numpy(), r["n_drafted"], err_msg=f"n_drafted, step {t}")
        np.testing.assert_array_equal(nr.cpu().numpy(), r["n_revoked"], err_msg=f"n_revoked, step {t}")
        for k in KEYS:
            np.testing.assert_array_equal(gst[k].cpu().numpy(), ost[k], err_msg=f"{k}, step {t}")
    return ost


@pytest.mark.parametrize("blk", [1, 32, 77, 256])
def test_revocable_runs_match_oracle(blk):
    st = _run(24, blk, 40, seed=blk, tau_replace=0.95, tau_draft=0.9, draft_budget=max(1, blk // 8), pi=0.7,
              cooldown=1, remask_budget=2, w_unc=1.0, w_infl=0.5, w_drift=2.0)
    assert st["masked"].sum() < st["masked"].size          # the runs make progress


def test_revocable_ties_and_no_budget():
    _run(16, 64, 30, seed=3, grid=8, tau_replace=0.875, tau_draft=0.75, draft_budget=0, pi=1.5, cooldown=0,
         remask_budget=3, w_unc=1.0, w_infl=1.0, w_drift=0.0)


def test_revocable_until_finished():
    # runs past the point where every sequence has finished: finished ones stay as they are
    st = _run(8, 16, 60, seed=5, tau_replace=0.99, tau_draft=0.5, draft_budget=4, pi=1.0, cooldown=1,
              remask_budget=1)
    assert st["masked"].sum() == 0


@pytest.mark.parametrize("blk,code,layout", [(32, "f16", "full"), (1, "f16", "full"), (100, "bf16", "full"),
                                             (256, "f16", "compact"), (77, "f32", "full")])
def test_attention_influence_matches_oracle(blk, code, layout):
    """dlm_attention_influence (the attention each block position receives
    from the masked queries, mean over layers and heads) against the oracle:
    full maps with the block inside and compact blocks, f16 / bf16 / f32
    attention, masks on both sides of DAPD's 50 % switch (the influence sums
    every sequence's masked rows whatever the fraction)."""
    import torch

    import diffusion_decoding_token_gb300 as dlm
    import synth
    from parity import close, to_torch
    rng = np.random.default_rng(blk)
    B, L, H = 5, 3, 4
    dt = {"f16": synth.F16, "bf16": synth.BF16, "f32": synth.F32}[code]
    sub = (rng.random((B, L, H, blk, blk)) ** 3 * 0.2).astype(np.float32)
    st = {synth.F32: lambda a: a, synth.BF16: synth.to_bf16_bits, synth.F16: synth.to_f16_bits}[dt](sub)
    bs = 0
    if layout == "full":
        bs = 16
        N = (bs + blk + 8 + 7) // 8 * 8
        full = np.zeros((B, L, H, N, N), st.dtype)
        full[:, :, :, bs:bs + blk, bs:bs + blk] = st
        st = full
    masked = (rng.random((B, blk)) < np.array([0.9, 0.6, 0.3, 0.0, 1.0])[:, None]).astype(np.uint8)
    status = dlm.new_status()
    g = dlm.attention_influence(to_torch(st, dt, "cuda"), torch.from_numpy(masked).cuda(), bs, status=status)
    o = oracle.attention_influence(st, masked, block_start=bs, dtype=None if dt == synth.F32 else dt)
    assert int(status.item()) == 0
    g = g.cpu().numpy()
    assert close(g, o, atol=1e-6, rtol=1e-6).all(), np.max(np.abs(g - o))
    assert (g[3] == 0).all()                                  # nothing masked: no influence
