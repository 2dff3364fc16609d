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

The static inputs come from ``synth.decode_problem``.  One step can be
captured in a CUDA graph and replayed (``run(graph=True)``).
"""
from __future__ import annotations

import numpy as np
import torch

from . import _binding as B


RULES = ("threshold", "factor", "topk", "cap", "dapd")


class SyntheticDecoder:
    def __init__(self, problem: dict, rule: str, device="cuda", *, tau=0.9, factor_f=1.0, topk_k=2,
                 tau_low=0.8, tau_high=0.95, gamma=-16.0, tau_edge=None, bulk_conf=0.9, bulk_frac=0.5,
                 max_steps=None):
        if rule not in RULES:
            raise ValueError(f"rule must be one of {RULES}")
        cfg = problem["cfg"]
        self.cfg, self.rule = cfg, rule
        dev = torch.device(device)
        self.dev = dev
        Bn, blk, V = cfg.batch, cfg.blk, cfg.vocab
        self.B, self.blk, self.V = Bn, blk, V
        self.max_steps = max_steps or blk
        f32 = dict(dtype=torch.float32, device=dev)
        self.logits = torch.from_numpy(problem["base"]).to(dev)
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

    def capture(self):
        """Capture one step as a CUDA graph (the buffers stay fixed)."""
        s = torch.cuda.Stream(device=self.dev)
        s.wait_stream(torch.cuda.current_stream(self.dev))
        saved = (self.tok.clone(), self.masked.clone(), self.steps.clone(), self.logits.clone())
        with torch.cuda.stream(s):
            self.step()  # warm-up outside the graph
        torch.cuda.current_stream(self.dev).wait_stream(s)
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph):
            self.step()
        torch.cuda.synchronize(self.dev)
        self.tok.copy_(saved[0])
        self.masked.copy_(saved[1])
        self.steps.copy_(saved[2])
        self.logits.copy_(saved[3])

    def run(self, graph: bool = False, check_every: int = 4, log=None):
        """Decode until nothing is masked (or max_steps); returns a summary.
        ``log``, a list, receives each step's selection (eager runs only)."""
        if graph and self.graph is None:
            self.capture()
        done_steps = 0
        while done_steps < self.max_steps:
            for _ in range(check_every if graph else 1):
                if graph:
                    self.graph.replay()
                else:
                    self.step()
                    if log is not None:
                        log.append(self.sel.cpu().numpy().copy())
                done_steps += 1
                if done_steps >= self.max_steps:
                    break
            if int(self.masked.sum().item()) == 0:
                break
        return self.summary()

    def summary(self) -> dict:
        tok = self.tok.cpu().numpy()
        target = self.target.view(self.B, self.blk).cpu().numpy()
        committed = tok >= 0
        wrong = committed & (tok != target)
        steps = self.steps.cpu().numpy()
        return dict(rule=self.rule, steps=steps, mean_steps=float(steps.mean()), tokens=tok,
                    error_rate=float(wrong.sum() / max(1, committed.sum())),
                    tokens_per_step=float(committed.sum() / max(1, steps.sum())),
                    unfinished=int((~committed).sum()), status=int(self.status.item()))
