"""Multi-step synthetic decode driver.

Runs the per-step decision path in a decoding loop over a deterministic
stand-in for the model, so the rules can be compared by the number of steps
(NFE) they need and by how often they commit a wrong token:

* model (stand-in for the forward pass; torch ops): every position i has a
  target token t_i and a decoy d_i.  With s_i the fraction of i's planted
  neighbours that are already decoded,
      z_i[t_i] = c0 + u_i + kappa * s_i,     z_i[d_i] = c0 + v_i * (1 - s_i),
  all other logits fixed background; c0 is the background's expected
  log-mass.  While its neighbours are masked a position may prefer its decoy;
  decoding them first makes the target win -- the dependency that parallel
  decoding can break (DAPD page, research motivation; Fast-dLLM review,
  "curse of parallel decoding").  The attention maps handed to DAPD are the
  planted graph's (static).
* step: model -> dlm_row_stats -> one selection rule -> commit the argmax
  token at every selected position (the caller's job in the library, done
  here with torch indexing).  A sequence counts a step while it still has a
  masked position.
* rule "revocable" (COVER page, revocable parallel decoding): the step is
  model -> dlm_row_stats (KL to the previous step = the seeds' drift) ->
  dlm_attention_influence (the attention each position receives from the
  masked queries) -> dlm_revocable_step, which verifies last step's seeds
  (the stand-in's prediction at a decoded position depends on its neighbours
  only, so it is a leave-one-out re-prediction), drafts masked positions and
  picks the next seeds.

The static inputs come from ``synth.decode_problem``.  The whole decode
(max_steps steps) can be captured as one CUDA graph and replayed
(``run(graph=True)``).
"""
from __future__ import annotations

import numpy as np
import torch

from . import _binding as B


RULES = ("threshold", "factor", "topk", "cap", "dapd", "revocable")


REVOCABLE_DEFAULT = dict(tau_replace=0.9, tau_draft=0.9, draft_budget=0, w_unc=1.0, w_infl=1.0, w_drift=1.0,
                         pi=1.0, cooldown=1, remask_budget=2)


class SyntheticDecoder:
    def __init__(self, problem: dict, rule: str, device="cuda", *, tau=0.9, factor_f=1.0, topk_k=2,
                 tau_low=0.8, tau_high=0.95, gamma=-16.0, tau_edge=None, bulk_conf=0.9, bulk_frac=0.5,
                 revocable=None, max_steps=None):
        if rule not in RULES:
            raise ValueError(f"rule must be one of {RULES}")
        cfg = problem["cfg"]
        self.cfg, self.rule = cfg, rule
        dev = torch.device(device)
        self.dev = dev
        Bn, blk, V = cfg.batch, cfg.blk, cfg.vocab
        self.B, self.blk, self.V = Bn, blk, V
        self.max_steps = max_steps or (3 * blk if rule == "revocable" else blk)
        f32 = dict(dtype=torch.float32, device=dev)
        self.logits = torch.from_numpy(problem["base"]).to(dev)
        self.base_logits = self.logits.clone() if rule == "revocable" else None
        self.rows = torch.arange(Bn * blk, device=dev)
        self.target = torch.from_numpy(problem["target"].reshape(-1)).to(dev)
        self.decoy = torch.from_numpy(problem["decoy"].reshape(-1)).to(dev)
        c0 = np.float32(problem["c0"])
        self.zt0 = torch.from_numpy((c0 + problem["u"]).astype(np.float32).reshape(-1)).to(dev)
        self.c0 = torch.tensor(c0, **f32)
        self.v = torch.from_numpy(problem["v"].reshape(-1)).to(dev)
        self.kappa = torch.tensor(np.float32(cfg.kappa), **f32)
        self.one = torch.tensor(np.float32(1.0), **f32)
        self.adj = torch.from_numpy(problem["links"].astype(np.int32)).to(dev)
        self.deg = self.adj.sum(-1).clamp(min=1).to(torch.float32).reshape(-1)
        self.attn = torch.from_numpy(problem["attn"].view(np.int16)).to(dev).view(torch.float16)
        self.tok = torch.full((Bn, blk), -1, dtype=torch.int32, device=dev)
        self.masked = torch.ones((Bn, blk), dtype=torch.uint8, device=dev)
        self.steps = torch.zeros(Bn, dtype=torch.int32, device=dev)
        self.status = B.new_status(dev)
        self.stats = B.alloc_row_stats(Bn * blk, dev, with_prev=False)
        self.sel = torch.zeros((Bn, blk), dtype=torch.uint8, device=dev)
        self.nsel = torch.zeros(Bn, dtype=torch.int32, device=dev)
        self.prm = dict(tau=tau, factor_f=factor_f, topk_k=topk_k, tau_low=tau_low, tau_high=tau_high, gamma=gamma,
                        tau_edge=cfg.tau_edge if tau_edge is None else tau_edge, bulk_conf=bulk_conf,
                        bulk_frac=bulk_frac)
        self.cap_ws = B.cap_workspace(Bn, blk, dev)
        self.dapd_ws = B.dapd_workspace(Bn, blk, dev)
        self.graph = None
        self.graph_steps = 0
        self.step_index = 0
        if rule == "revocable":
            # seeds' cache drift = KL to the previous step's distribution; downstream
            # influence = attention received from masked queries, mean over layers x heads
            # (dlm_attention_influence)
            self.rev = dict(REVOCABLE_DEFAULT, **(revocable or {}))
            self.state = B.revocable_state(Bn, blk, dev)
            self.tok, self.masked = self.state["tok"], self.state["masked"]
            self.prev_logits = self.logits.clone()
            self.stats = B.alloc_row_stats(Bn * blk, dev, with_prev=True)
            self.infl = torch.zeros((Bn, blk), dtype=torch.float32, device=dev)
            self.outcome = torch.zeros((Bn, blk), dtype=torch.uint8, device=dev)
            self.n_revised = torch.zeros(Bn, dtype=torch.int32, device=dev)

    # -- the stand-in model ------------------------------------------------
    def model(self):
        decoded = (self.masked == 0).to(torch.int32)                       # [B, blk]
        cnt = (self.adj * decoded[:, None, :]).sum(-1).reshape(-1)          # exact counts
        s = cnt.to(torch.float32) / self.deg                               # fp32, IEEE division
        zt = self.zt0 + self.kappa * s
        zd = self.c0 + self.v * (self.one - s)
        self.logits[self.rows, self.target] = zt
        self.logits[self.rows, self.decoy] = zd

    # -- one decoding step ---------------------------------------------------
    def step(self):
        Bn, blk = self.B, self.blk
        active = (self.masked.sum(-1) > 0).to(torch.int32)
        self.steps += active
        self.model()
        if self.rule == "revocable":
            self._revocable_step()
            return
        st = B.row_stats(self.logits, out=self.stats, status=self.status)
        conf = st.conf.view(Bn, blk)
        p = self.prm
        if self.rule == "threshold":
            B.select_threshold(conf, self.masked, p["tau"], selected=self.sel, n_selected=self.nsel)
        elif self.rule == "factor":
            B.select_factor(conf, self.masked, p["factor_f"], selected=self.sel, n_selected=self.nsel)
        elif self.rule == "topk":
            B.select_topk(conf, self.masked, p["topk_k"], selected=self.sel, n_selected=self.nsel)
        elif self.rule == "cap":
            B.cap_select(self.logits, st.argmax.view(Bn, blk), conf, st.lse.view(Bn, blk), self.masked,
                         p["tau_low"], p["tau_high"], p["gamma"], blk, workspace=self.cap_ws, status=self.status,
                         selected=self.sel, n_selected=self.nsel)
        else:
            B.dapd_graph_mis(self.attn, self.masked, conf, p["tau_edge"], p["bulk_conf"], p["bulk_frac"], 0, 0,
                             workspace=self.dapd_ws, status=self.status, selected=self.sel, n_selected=self.nsel)
        chosen = self.sel.to(torch.bool)
        self.tok.copy_(torch.where(chosen, st.argmax.view(Bn, blk), self.tok))
        self.masked.mul_((~chosen).to(torch.uint8))

    def _revocable_step(self):
        Bn, blk = self.B, self.blk
        st = B.row_stats(self.logits, self.prev_logits, out=self.stats, status=self.status)
        self.prev_logits.copy_(self.logits)
        infl = B.attention_influence(self.attn, self.masked, 0, out=self.infl, workspace=self.dapd_ws,
                                     status=self.status)
        r = self.rev
        B.revocable_step(st.argmax.view(Bn, blk), st.conf.view(Bn, blk), self.state, self.step_index,
                         tau_replace=r["tau_replace"], tau_draft=r["tau_draft"], draft_budget=r["draft_budget"],
                         w_unc=r["w_unc"], w_infl=r["w_infl"], w_drift=r["w_drift"], pi=r["pi"],
                         cooldown=r["cooldown"], remask_budget=r["remask_budget"], influence=infl,
                         drift=st.kl.view(Bn, blk), outcome=self.outcome, n_drafted=self.nsel)
        self.sel.copy_(self.outcome)
        self.n_revised += (self.outcome >= 3).sum(-1, dtype=torch.int32)
        self.step_index += 1

    def capture(self, n_steps: int | None = None):
        """Capture ``n_steps`` decoding steps (default: the whole decode,
        max_steps of them) as one CUDA graph.  A sequence with nothing masked
        selects nothing and counts no step, so the surplus steps of a
        finished sequence change nothing."""
        n_steps = self.max_steps if n_steps is None else n_steps
        s = torch.cuda.Stream(device=self.dev)
        s.wait_stream(torch.cuda.current_stream(self.dev))
        saved = (self.tok.clone(), self.masked.clone(), self.steps.clone(), self.logits.clone())
        with torch.cuda.stream(s):
            self.step()  # warm-up outside the graph
        torch.cuda.current_stream(self.dev).wait_stream(s)
        self.step_index = 0  # the captured steps carry step indices 0 .. n_steps-1
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph):
            for _ in range(n_steps):
                self.step()
        torch.cuda.synchronize(self.dev)
        self.graph_steps = n_steps
        self.reset(saved)

    def reset(self, saved=None):
        """Back to the initial state (everything masked, nothing committed)."""
        if saved is None:
            self.tok.fill_(-1)
            self.masked.fill_(1)
            self.steps.zero_()
        else:
            self.tok.copy_(saved[0])
            self.masked.copy_(saved[1])
            self.steps.copy_(saved[2])
            self.logits.copy_(saved[3])
        self.step_index = 0
        if self.rule == "revocable":
            self.state["seed"].zero_()
            self.state["last_seed"].fill_(-(2 ** 30))
            self.state["remasks"].zero_()
            self.state["last_tok"].fill_(-1)
            self.state["flipflops"].zero_()
            self.n_revised.zero_()
            self.prev_logits.copy_(self.base_logits)

    def run(self, graph: bool = False, log=None):
        """Decode until nothing is masked (or max_steps); returns a summary.
        ``graph``: replay the captured whole-decode graph (captured on first
        use).  ``log``, a list, receives each step's selection (eager runs)."""
        if graph:
            if self.graph is None:
                self.capture()
            self.graph.replay()
            return self.summary()
        for _ in range(self.max_steps):
            self.step()
            if log is not None:
                log.append(self.sel.cpu().numpy().copy())
            if int(self.masked.sum().item()) == 0:
                break
        return self.summary()

    def summary(self) -> dict:
        tok = self.tok.cpu().numpy()
        target = self.target.view(self.B, self.blk).cpu().numpy()
        committed = tok >= 0
        wrong = committed & (tok != target)
        steps = self.steps.cpu().numpy()
        out = dict(rule=self.rule, steps=steps, mean_steps=float(steps.mean()), tokens=tok,
                   error_rate=float(wrong.sum() / max(1, committed.sum())),
                   tokens_per_step=float(committed.sum() / max(1, steps.sum())),
                   unfinished=int((~committed).sum()), status=int(self.status.item()))
        if self.rule == "revocable":
            out["revisions"] = int(self.n_revised.sum().item())
            out["remasks"] = int(self.state["remasks"].sum().item())
            out["flipflops"] = int(self.state["flipflops"].sum().item())
        return out


class DepCapDecoder:
    """DepCap's block loop over a whole generation (DepCap, "Methodology"):
    DepGA-Block picks each block's length from the change in KL that the last
    decoded block caused in the window of future positions, against their
    entropy; CAP-Decoding then unmasks a conflict-free subset of the block
    per step until the block is done.

    The problem's ``cfg.blk`` is the generation length N.  Per step, for every
    sequence b with cursor_b (its first undecoded position):

    1. model over all N positions (as in :class:`SyntheticDecoder`);
    2. the window rows are rows b*N + cursor_b + k, k < L_max, of the
       generation's logits (positions past the end repeat the last one and
       are never used), named by a row index -- nothing is copied;
    3. ``dlm_row_stats_ex`` in gather mode over those rows against the same
       rows of the snapshot -> ŷ, c, LSE, H, KL at window slot b*L_max + k;
    4. sequences without a block: ``dlm_depcap_boundary_ragged`` with
       L_window = min(L_max, N - cursor_b) (cold start for the first block)
       sets the block length, and this forward pass becomes the sequence's
       snapshot, the "before" of the next boundary's KL;
    5. ``dlm_cap_select`` over the window (the same row index) with scope =
       the block length;
    6. commit ŷ at the selected positions; a block with nothing masked left
       advances the cursor.

    The stand-in model rewrites only the target and decoy logit of each row
    (the background never changes), so taking a sequence's snapshot copies
    those two entries of its rows; the snapshot equals a full copy of the
    forward pass's logits.

    Reading: p_prev of the KL is the model's distribution at the forward pass
    where the last block began (before any of its tokens were committed),
    p_curr the one after its last commit.
    """

    def __init__(self, problem: dict, device="cuda", *, L_max=32, lam=1.2, L_min=8, smooth_w=1, norm_mode=0,
                 tau_low=0.8, tau_high=0.95, gamma=-16.0, max_steps=None):
        cfg = problem["cfg"]
        dev = torch.device(device)
        Bn, N, V = cfg.batch, cfg.blk, cfg.vocab
        if not 1 <= L_max <= min(N, B.MAX_BLK):
            raise ValueError("L_max must be in [1, min(N, 256)]")
        self.cfg, self.dev, self.B, self.N, self.V, self.L_max = cfg, dev, Bn, N, V, L_max
        self.max_steps = max_steps or N
        self.prm = dict(lam=lam, L_min=L_min, smooth_w=smooth_w, norm_mode=norm_mode, tau_low=tau_low,
                        tau_high=tau_high, gamma=gamma)
        f32 = dict(dtype=torch.float32, device=dev)
        i32 = dict(dtype=torch.int32, device=dev)
        self.logits = torch.from_numpy(problem["base"]).to(dev)               # [B*N, V]
        self.snapshot = self.logits.clone()
        self.rows = torch.arange(Bn * N, device=dev)
        self.target = torch.from_numpy(problem["target"].reshape(-1)).to(dev)
        self.decoy = torch.from_numpy(problem["decoy"].reshape(-1)).to(dev)
        c0 = np.float32(problem["c0"])
        self.zt0 = torch.from_numpy((c0 + problem["u"]).astype(np.float32).reshape(-1)).to(dev)
        self.c0 = torch.tensor(c0, **f32)
        self.v = torch.from_numpy(problem["v"].reshape(-1)).to(dev)
        self.kappa = torch.tensor(np.float32(cfg.kappa), **f32)
        self.one = torch.tensor(np.float32(1.0), **f32)
        self.adj = torch.from_numpy(problem["links"].astype(np.int32)).to(dev)
        self.deg = self.adj.sum(-1).clamp(min=1).to(torch.float32).reshape(-1)
        self.k = torch.arange(L_max, **i32)
        self.seq = torch.arange(Bn, device=dev)
        self.tok = torch.full((Bn, N), -1, **i32)
        self.masked = torch.ones((Bn, N), dtype=torch.uint8, device=dev)
        self.cursor = torch.zeros(Bn, **i32)
        self.blen = torch.zeros(Bn, **i32)           # 0: the next step picks a new block
        self.cold = torch.ones(Bn, dtype=torch.uint8, device=dev)
        self.steps = torch.zeros(Bn, **i32)
        self.n_blocks = torch.zeros(Bn, **i32)
        self.status = B.new_status(dev)
        self.stats = B.alloc_row_stats(Bn * L_max, dev, with_prev=True)
        self.new_len = torch.zeros(Bn, **i32)
        self.score = torch.zeros((Bn, L_max), **f32)
        self.sel = torch.zeros((Bn, L_max), dtype=torch.uint8, device=dev)
        self.nsel = torch.zeros(Bn, **i32)
        self.cap_ws = B.cap_workspace(Bn, L_max, dev)
        self.graph = None
        self.graph_steps = 0
        self.trace = None

    def model(self):
        decoded = (self.masked == 0).to(torch.int32)
        cnt = (self.adj * decoded[:, None, :]).sum(-1).reshape(-1)
        s = cnt.to(torch.float32) / self.deg
        zt = self.zt0 + self.kappa * s
        zd = self.c0 + self.v * (self.one - s)
        self.logits[self.rows, self.target] = zt
        self.logits[self.rows, self.decoy] = zd

    def step(self):
        Bn, N, Lm = self.B, self.N, self.L_max
        p = self.prm
        active = self.cursor < N
        self.steps += active.to(torch.int32)
        self.model()
        pos = (self.cursor[:, None] + self.k[None, :]).clamp(max=N - 1)               # [B, L_max]
        row_index = (self.seq[:, None] * N + pos).reshape(-1).to(torch.int32)
        window_len = (N - self.cursor).clamp(min=0, max=Lm)
        st = B.row_stats(self.logits, self.snapshot, row_index=row_index, gather=True, out=self.stats,
                         status=self.status)
        need = active & (self.blen == 0)
        B.depcap_boundary(st.kl.view(Bn, Lm), st.entropy.view(Bn, Lm), p["lam"], p["L_min"], p["smooth_w"],
                          p["norm_mode"], cold_start=self.cold, window_len=window_len, block_len=self.new_len,
                          score=self.score)
        self.blen.copy_(torch.where(need, self.new_len, self.blen))
        self.n_blocks += need.to(torch.int32)
        self.cold.mul_((~need).to(torch.uint8))
        needv = need.repeat_interleave(N)
        for tok in (self.target, self.decoy):
            now = self.logits[self.rows, tok]
            self.snapshot[self.rows, tok] = torch.where(needv, now, self.snapshot[self.rows, tok])
        in_block = self.k[None, :] < self.blen[:, None]
        mwin = (torch.gather(self.masked, 1, pos.to(torch.int64)) * in_block.to(torch.uint8)).contiguous()
        B.cap_select(self.logits, st.argmax.view(Bn, Lm), st.conf.view(Bn, Lm), st.lse.view(Bn, Lm), mwin,
                     p["tau_low"], p["tau_high"], p["gamma"], Lm, scope_len=self.blen, workspace=self.cap_ws,
                     status=self.status, selected=self.sel, n_selected=self.nsel, row_index=row_index)
        if self.trace is not None:
            self.trace.append(dict(cursor=self.cursor.cpu().numpy(), need=need.cpu().numpy(),
                                   blen=self.blen.cpu().numpy(), sel=self.sel.cpu().numpy(),
                                   masked=self.masked.cpu().numpy()))
        # commit: the selected positions are distinct (k < blen <= window), so
        # accumulating into zeros writes each at most once
        chosen = self.sel.to(torch.int32)
        flat = (self.seq[:, None] * N + pos).reshape(-1)
        dec = torch.zeros(Bn * N, dtype=torch.int32, device=self.dev)
        dec.index_put_((flat,), chosen.reshape(-1), accumulate=True)
        val = torch.zeros(Bn * N, dtype=torch.int32, device=self.dev)
        val.index_put_((flat,), (chosen * st.argmax.view(Bn, Lm)).reshape(-1), accumulate=True)
        dec = dec.view(Bn, N) > 0
        self.tok.copy_(torch.where(dec, val.view(Bn, N), self.tok))
        self.masked.mul_((~dec).to(torch.uint8))
        left = (torch.gather(self.masked, 1, pos.to(torch.int64)) * in_block.to(torch.uint8)).sum(-1)
        done = active & (self.blen > 0) & (left == 0)
        self.cursor.copy_(torch.where(done, self.cursor + self.blen, self.cursor))
        self.blen.copy_(torch.where(done, torch.zeros_like(self.blen), self.blen))

    def capture(self, n_steps: int | None = None):
        """Capture ``n_steps`` steps (default: max_steps, the whole decode) as
        one CUDA graph; a finished sequence's surplus steps change nothing."""
        n_steps = self.max_steps if n_steps is None else n_steps
        s = torch.cuda.Stream(device=self.dev)
        s.wait_stream(torch.cuda.current_stream(self.dev))
        with torch.cuda.stream(s):
            self.step()
        torch.cuda.current_stream(self.dev).wait_stream(s)
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph):
            for _ in range(n_steps):
                self.step()
        torch.cuda.synchronize(self.dev)
        self.graph_steps = n_steps
        self.reset()

    def reset(self):
        self.tok.fill_(-1)
        self.masked.fill_(1)
        self.cursor.zero_()
        self.blen.zero_()
        self.cold.fill_(1)
        self.steps.zero_()
        self.n_blocks.zero_()

    def run(self, graph: bool = False, trace: bool = False):
        """Decode the whole generation; ``trace`` records every step's state
        (eager runs only)."""
        if graph:
            if self.graph is None:
                self.capture()
            self.graph.replay()
            return self.summary()
        self.trace = [] if trace else None
        for _ in range(self.max_steps):
            self.step()
            if bool((self.cursor >= self.N).all()):
                break
        return self.summary()

    def summary(self) -> dict:
        tok = self.tok.cpu().numpy()
        target = self.target.view(self.B, self.N).cpu().numpy()
        committed = tok >= 0
        steps = self.steps.cpu().numpy()
        return dict(rule="depcap", steps=steps, mean_steps=float(steps.mean()), tokens=tok,
                    n_blocks=self.n_blocks.cpu().numpy(),
                    error_rate=float((committed & (tok != target)).sum() / max(1, committed.sum())),
                    tokens_per_step=float(committed.sum() / max(1, steps.sum())),
                    unfinished=int((~committed).sum()), status=int(self.status.item()), trace=self.trace)
