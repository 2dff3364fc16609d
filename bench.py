"""Benchmark of the per-step unmask-decision hot path on GB300.

One "step" = the whole path over one batch: the fused row-statistics pass over
every masked position's current and previous logit rows, then the four
selection rules (Fast-dLLM threshold, DepGA-Block boundary, CAP-Decoding,
DAPD graph + Welsh-Powell) for every sequence.

Workload (batched serving): 64 independent sequences x 32 masked positions,
vocab 152064, bf16 current and previous logits (1.25 GB per step, larger than
L2, so no flush is needed between steps), fp16 attention 10 layers x 28 heads
over 512 positions.  Inputs are synthetic (``synth``), seeded, and resident in
HBM before the timed region.

Prints one JSON line: decisions/s (masked positions decided per second, all
ranks), the row pass's achieved HBM bandwidth against the measured peak, the
end-to-end number through host buffers, the SM clocks seen, and the fp64 CPU
oracle timed on a bounded sample.  ``--impl reference`` times the oracle
itself as the reference arm.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "masked-position decisions/sec per decode step; logit-read GB/s vs HBM peak"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--seed", type=int, default=1004)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=5)
    ap.add_argument("--serial-dapd", action="store_true",
                    help="run the DAPD chain on the main stream after the other rules (default: on a side stream)")
    ap.add_argument("--late-dapd-fork", action="store_true",
                    help="fork the DAPD chain after the row pass (default: the attention graph starts with the "
                         "step on the low-priority side stream and takes the SMs the row pass's last wave leaves "
                         "free; the selection waits for the statistics)")
    ap.add_argument("--dapd-priority", default="low", choices=["low", "high"],
                    help="priority of the DAPD side stream (high: the attention pass takes SMs from the step's "
                         "start and the row pass shares them)")
    ap.add_argument("--flush-l2", default="auto", choices=["auto", "on", "off"],
                    help="write a 512 MB buffer between timed steps (auto: when a step reads less than twice L2)")
    ap.add_argument("--serial-rules", action="store_true",
                    help="run threshold, boundary and CAP one after another (default: parallel graph branches)")
    ap.add_argument("--whole-graph", action="store_true",
                    help="capture every timed step (row pass, DAPD chain, rules) in CUDA graphs, the row-pass "
                         "timing events as event nodes inside them (default: the row pass and the DAPD chain "
                         "launched each step, the rules replayed as one captured graph; measured faster: the "
                         "event nodes and cross-stream edges of a captured step add latency between kernels)")
    ap.add_argument("--rules-graph", action="store_true", help="the default (kept for older command lines)")
    ap.add_argument("--no-graph", action="store_true",
                    help="launch the rules eagerly instead of replaying them as one captured CUDA graph")
    ap.add_argument("--extra-rules", default="",
                    help="comma list of extra selection rules to run in every step: topk, factor")
    ap.add_argument("--workload", default="batched",
                    help="batched (default, the headline), tiny, llada_step, depcap_window, stress_graph, stress_bulk")
    ap.add_argument("--driver", action="store_true",
                    help="instead of the step benchmark: whole synthetic decodes per rule (steps/NFE, error rate, "
                         "decode time as one CUDA graph)")
    ap.add_argument("--boost-mode", default="relative", choices=["relative", "absolute"],
                    help="logit boost reading of the input recipe (absolute = literal: no confidence reaches the "
                         "thresholds; the bytes are the same)")
    ap.add_argument("--batch", type=int, default=0, help="override the sequences per GPU (small profiling cases)")
    ap.add_argument("--fuse-rules", default="auto", choices=["auto", "on", "off"],
                    help="run threshold, boundary and CAP inside the row pass (dlm_row_stats_rules); auto: only the "
                         "DepCap chain (boundary -> CAP, no DAPD)")
    ap.add_argument("--fold-attention", default="auto", choices=["auto", "off"],
                    help="compute the DAPD attention sums in the row pass's own CTAs (dlm_row_stats_attention) "
                         "where the library can; off: a separate attention pass on the side stream")
    ap.add_argument("--no-per-workload", action="store_true",
                    help="skip the short runs of the other workloads after the headline one")
    ap.add_argument("--per-workload-steps", type=int, default=200,
                    help="timed steps of each other workload in the per_workload block")
    ap.add_argument("--compact-attn", action="store_true",
                    help="hold only the attention block [B, L, H, blk, blk] on the device (small profiling cases)")
    return ap.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def workload_desc(cfg):
    dt = {0: "f32", 1: "bf16", 2: "f16"}
    m = cfg.blk if cfg.masked_count < 0 else cfg.masked_count
    att = (f", {dt[cfg.attn_dtype]} attention {cfg.n_layers}x{cfg.n_heads} over {cfg.seq_len} positions"
           if cfg.n_layers else "")
    return (f"{cfg.name}: B={cfg.batch} sequences x {m} masked of {cfg.blk} positions, V={cfg.vocab} "
            f"{dt[cfg.logit_dtype]} current+previous logits{att}; rules: {', '.join(cfg.rules)}")


def row_pass_bytes(cfg, w, rows, folded):
    """Algorithmic bytes of one row pass: the current and previous logit rows
    it reads, plus, when the DAPD attention sums are folded into it, the
    attention runs of the masked rows of sequences on the graph path."""
    import synth
    esz = 4 if cfg.logit_dtype == synth.F32 else 2
    b = 2 * rows * cfg.vocab * esz
    if folded:
        asz = 4 if cfg.attn_dtype == synth.F32 else 2
        m = w.masked.sum(axis=1)
        graph = m >= cfg.bulk_frac * cfg.blk
        b += cfg.n_layers * cfg.n_heads * int((m * graph).sum()) * cfg.blk * asz
    return b


def recorded_traffic():
    """DRAM bytes per row-pass launch from the committed ncu summary, valid
    only while the kernel source still matches the one that was profiled."""
    import hashlib
    summary = os.path.join(ROOT, "profiles", "row_stats_batched.md")
    src = os.path.join(ROOT, "diffusion_decoding_token_gb300", "csrc", "row_stats.cu")
    if not (os.path.exists(summary) and os.path.exists(src)):
        return None
    kv = {}
    for line in open(summary):
        if ":" in line and line.split(":")[0].strip() in ("traffic_bytes_per_launch", "kernel_source_sha256_16"):
            k, v = line.split(":", 1)
            kv[k.strip()] = v.strip()
    h = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    if kv.get("kernel_source_sha256_16") != h or "traffic_bytes_per_launch" not in kv:
        return None
    return int(kv["traffic_bytes_per_launch"])


def device_info(local):
    """GPU name, SM count, CUDA runtime and driver versions of this rank's GPU."""
    import torch
    p = torch.cuda.get_device_properties(local)
    info = {"name": p.name, "sm_count": p.multi_processor_count, "cuda_runtime": torch.version.cuda,
            "torch": torch.__version__}
    try:
        out = subprocess.run(["nvidia-smi", "--query-gpu=driver_version", "--format=csv,noheader", "-i", str(local)],
                             capture_output=True, text=True, timeout=20)
        if out.returncode == 0:
            info["driver"] = out.stdout.strip()
    except (OSError, subprocess.SubprocessError):
        pass
    return info


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during the timed region."""

    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self, window=None):
        """Median SM clock and throttle reasons of the samples taken inside
        ``window`` (host wall-clock interval of the timed region) -- or, if
        the region was shorter than a few sampling periods, of the load phase
        run just before it."""
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        lines = self.lines
        inside = [x for x in lines if window and window[0] <= x[0] <= window[1]]
        used = "timed region"
        if len(inside) >= 3:
            lines = inside
        else:
            used = "load phase + timed region"
        for _, ln in lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm), "window": used}


# ------------------------------------------------------------ multi-rank
def max_over_ranks(x: float, world: int, device=None) -> float:
    """The maximum of a per-rank scalar over all ranks (identity at N=1).
    Only a timing scalar crosses ranks: the decision path has no collective."""
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as td
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    td.all_reduce(t, op=td.ReduceOp.MAX)
    return float(t.item())


def job_throughput(decisions_per_rank_step: int, world: int, steps: int, max_ms: float) -> float:
    """Whole-job decisions/s: every rank decides its own batch each step
    (weak scaling), timed by the slowest rank."""
    return decisions_per_rank_step * world * steps / (max_ms / 1000.0)


# ------------------------------------------------------------------ native
def bench_config(args):
    import synth
    cfg = synth.CONFIGS[args.workload]
    if args.batch:
        cfg = synth.scaled(cfg, batch=args.batch)
    if args.boost_mode != cfg.boost_mode:
        cfg = synth.scaled(cfg, boost_mode=args.boost_mode)
    return cfg


def run_native(args, rank, world, local, light=False):
    """The timed steps of one workload.  ``light``: only the timed steps of
    the full path (no per-rule runs, no attention-alone timing, no end-to-end
    steps, no clock sampling) -- the short runs of the per_workload block."""
    import torch

    import diffusion_decoding_token_gb300 as dlm
    import synth

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    cfg = bench_config(args)
    B, blk, V = cfg.batch, cfg.blk, cfg.vocab
    w = synth.make(cfg, seed=args.seed + 100 * rank)
    tdt = {synth.F32: torch.float32, synth.BF16: torch.bfloat16, synth.F16: torch.float16}

    def dev_of(a, code):
        if code == synth.F32:
            return torch.from_numpy(a).to(dev)
        return torch.from_numpy(a.view(np.int16)).to(dev).view(tdt[code])

    cur = dev_of(w.cur, cfg.logit_dtype)
    prev = dev_of(w.prev, cfg.logit_dtype)
    masked = torch.from_numpy(w.masked).to(dev)
    row_index = None
    if cfg.masked_count >= 0:
        row_index = torch.from_numpy(np.nonzero(w.masked.reshape(-1))[0].astype(np.int32)).to(dev)
    N, bs = cfg.seq_len, cfg.block_start
    attn = None
    if cfg.n_layers and args.compact_attn:
        attn, bs = dev_of(w.attn, cfg.attn_dtype), 0
    elif cfg.n_layers:
        attn = torch.zeros((B, cfg.n_layers, cfg.n_heads, N, N), dtype=tdt[cfg.attn_dtype], device=dev)
        attn[:, :, :, bs:bs + blk, bs:bs + blk] = dev_of(w.attn, cfg.attn_dtype)

    status = dlm.new_status(dev)
    # the step runs on a high-priority stream so the DAPD side stream (lowest
    # priority) only takes SMs the row pass leaves free
    torch.cuda.synchronize()
    lo, hi = torch.cuda.Stream.priority_range()
    # the row pass's stream outranks the DAPD side stream (or, with
    # --dapd-priority high, is outranked by it)
    torch.cuda.set_stream(torch.cuda.Stream(device=dev, priority=lo if args.dapd_priority == "high" else hi))
    stream = torch.cuda.current_stream(dev)
    common = dict(tau=cfg.tau, lam=cfg.lam, L_min=cfg.L_min, tau_low=cfg.tau_low, tau_high=cfg.tau_high,
                  gamma=cfg.gamma, p_max=cfg.p_max, tau_edge=cfg.tau_edge, bulk_conf=cfg.bulk_conf,
                  bulk_frac=cfg.bulk_frac, status=status)
    extra = tuple(r for r in args.extra_rules.split(",") if r)
    common.update(rules=tuple(cfg.rules) + extra, cap_scope_from_boundary=(cfg.name == "depcap_window"),
                  concurrent_dapd=not args.serial_dapd, dapd_early=not args.late_dapd_fork, dapd_priority=args.dapd_priority,
                  parallel_rules=not args.serial_rules,
                  fuse_rules={"auto": "auto", "on": True, "off": False}[args.fuse_rules],
                  fold_attention="auto" if args.fold_attention == "auto" else False)
    plan = dlm.StepPlan(cur, prev, masked, attn=attn, block_start=bs, row_index=row_index, **common)

    for _ in range(args.warmup):
        plan.run(stream)
    torch.cuda.synchronize()
    # the rules (everything after the row pass) as one CUDA graph; the row
    # pass stays an eager launch so CUDA events can bracket it every step
    rules_graph = None
    if not args.no_graph and plan.has_rules_after_rows:
        rules_graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(rules_graph, stream=stream):
            plan.run(rules_only=True)
        torch.cuda.synchronize()

    def run_step(ev=None):
        if rules_graph is None:
            plan.run(stream, events=ev)
            return
        plan.run_rows(stream, events=ev)
        rules_graph.replay()
        plan.join(stream)

    for _ in range(args.warmup):
        run_step()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()

    esz = 4 if cfg.logit_dtype == synth.F32 else 2
    step_bytes = 2 * int(w.masked.sum()) * cfg.vocab * esz
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = args.flush_l2 == "on" or (args.flush_l2 == "auto" and step_bytes < 2 * l2)
    scrub = torch.empty(512 << 20, dtype=torch.uint8, device=dev) if flush else None
    whole = args.whole_graph and not args.no_graph
    # timing events; inside a captured graph they are external event nodes
    ev_kw = dict(enable_timing=True, external=True) if whole else dict(enable_timing=True)
    evs = [[torch.cuda.Event(**ev_kw) for _ in range(2)] for _ in range(args.steps)]
    s_ev = [(torch.cuda.Event(**ev_kw), torch.cuda.Event(**ev_kw)) for _ in range(args.steps)] if flush else None

    def timed_step(k):
        if flush:
            # each step timed on its own, with a 512 MB write before it (not timed)
            scrub.fill_(k & 0xff)
            s_ev[k][0].record(stream)
        if whole:
            plan.run(stream, events=evs[k])
        else:
            run_step(evs[k])
        if flush:
            s_ev[k][1].record(stream)

    step_graphs = []
    if whole:
        # the timed steps, captured back to back (at most 250 per graph):
        # every kernel of every step runs, with no host launch between them
        for c0 in range(0, args.steps, 250):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for k in range(c0, min(args.steps, c0 + 250)):
                    timed_step(k)
            step_graphs.append(g)
        torch.cuda.synchronize()
        step_graphs[0].replay()  # upload / warm-up (untimed)
        torch.cuda.synchronize()

    sampler = ClockSampler(local) if rank == 0 and not light else None
    if sampler:
        sampler.start()
        # load phase (untimed): keeps the GPU busy for ~1 s so the clock
        # samples reflect the clocks under this load
        t_end = time.time() + 1.0
        while time.time() < t_end:
            for _ in range(50):
                run_step()
            torch.cuda.synchronize()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    w0 = time.time()
    t0.record(stream)
    if whole:
        for g in step_graphs:
            g.replay()
    else:
        for k in range(args.steps):
            timed_step(k)
    t1.record(stream)
    host_ms = (time.time() - w0) * 1000.0 / args.steps
    torch.cuda.synchronize()
    w1 = time.time()
    if world > 1:
        torch.distributed.barrier()
    clocks = sampler.stop((w0, w1)) if sampler else None
    total_ms = sum(a.elapsed_time(b) for a, b in s_ev) if flush else t0.elapsed_time(t1)
    del step_graphs
    k1 = [e[0].elapsed_time(e[1]) for e in evs]
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())} during the benchmark")
    if light:
        return dict(total_ms=total_ms, k1=k1, flush=flush, cfg=cfg, w=w, decisions=int(w.masked.sum()),
                    rows=int(w.masked.sum()), launches=plan.n_launches * args.steps, fused=list(plan.fused),
                    folded=plan.folded)

    # the four rules alone, on the statistics of the last step
    r0 = torch.cuda.Event(enable_timing=True)
    r1 = torch.cuda.Event(enable_timing=True)
    for _ in range(3):
        rules_graph.replay() if rules_graph is not None else plan.run(stream, rules_only=True)
    r0.record(stream)
    for _ in range(100):
        rules_graph.replay() if rules_graph is not None else plan.run(stream, rules_only=True)
    r1.record(stream)
    torch.cuda.synchronize()
    rules_ms = r0.elapsed_time(r1) / 100

    def time_steps(p, n):
        """ms per step of plan p: eager row pass + its rules as one graph, each
        step alone after the scrub write when the inputs fit in L2."""
        p.run(stream)
        torch.cuda.synchronize()
        g = None
        if p.has_rules_after_rows:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                p.run(rules_only=True)
            torch.cuda.synchronize()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
        for k in range(n + 3):
            if flush:
                scrub.fill_(k & 0xff)
            if k >= 3:
                ev[k - 3][0].record(stream)
            p.run_rows(stream)
            if g is not None:
                g.replay()
            p.join(stream)
            if k >= 3:
                ev[k - 3][1].record(stream)
        torch.cuda.synchronize()
        return sum(a.elapsed_time(b) for a, b in ev) / n

    # each rule with the row pass, and the row pass alone (decisions/s per rule)
    per_rule = {}
    n_rule = max(20, min(300, args.steps))
    for rules in [()] + [(r,) for r in plan.rules]:
        kw = dict(common, rules=rules, concurrent_dapd=("dapd" in rules) and not args.serial_dapd)
        p = dlm.StepPlan(cur, prev, masked, attn=attn, block_start=bs, row_index=row_index, **kw)
        ms = time_steps(p, n_rule)
        per_rule["+".join(rules) or "row_pass_only"] = {"decisions_per_s": int(w.masked.sum()) * world / (ms / 1e3),
                                                         "ms_per_step": ms}
        del p

    # the DAPD attention graph alone (K6): attention GB/s.  The block's
    # attention can fit in L2 (36.7 MB on the batched workload) while in a step
    # it is read cold, so L2 is flushed before every timed pass here
    attention = None
    if "dapd" in plan.rules:
        ws = dlm.dapd_workspace(B, blk, dev)
        a_scrub = scrub if scrub is not None else torch.empty(512 << 20, dtype=torch.uint8, device=dev)
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(100)]
        for k in range(103):
            a_scrub.fill_(k & 0xff)
            if k >= 3:
                ev[k - 3][0].record(stream)
            dlm.dapd_graph(attn, masked, cfg.tau_edge, cfg.bulk_conf, cfg.bulk_frac, 0, bs, workspace=ws,
                           status=status)
            if k >= 3:
                ev[k - 3][1].record(stream)
        torch.cuda.synchronize()
        a_ms = sum(x.elapsed_time(y) for x, y in ev) / 100
        asz = 4 if cfg.attn_dtype == synth.F32 else 2
        # only the masked rows of the block are read: L * H * M * blk elements per sequence
        a_bytes = cfg.n_layers * cfg.n_heads * int(w.masked.sum()) * blk * asz
        attention = {"gbps": a_bytes / (a_ms / 1e3) / 1e9, "ms": a_ms, "algorithmic_bytes": a_bytes,
                     "kernels": "dapd_accum + dapd_graph, alone on the GPU, L2 flushed before each pass"}
        del a_scrub

    # --- end to end through host buffers (pinned), same public API.  Each step
    # uploads its new logits, its attention block and its mask, decides, and
    # reads the selections back.  As in a decode loop, the previous step's
    # logits are the previous step's upload and stay resident as `prev`.  The
    # uploads are pipelined: three device sets rotate (step k reads logits
    # D[k % 3] as cur and D[(k - 1) % 3] as prev, with attention and mask set
    # k % 3), and step k+1's upload runs on a copy stream while step k
    # decides, after step k-1 -- the last reader of the set it overwrites --
    # has finished.  Every step's copies are inside the timed region.
    e2e = None
    if args.e2e_steps > 0:
        NB = 3
        host_rows = [t.cpu().pin_memory() for t in (cur, prev, cur)]
        attn_h = None if w.attn is None else (torch.from_numpy(w.attn) if cfg.attn_dtype == synth.F32 else
                                              torch.from_numpy(w.attn.view(np.int16)).view(tdt[cfg.attn_dtype]))
        attn_h = None if attn_h is None else attn_h.pin_memory()
        masked_h = torch.from_numpy(w.masked).pin_memory()
        dev_rows = [cur.clone() for _ in range(NB)]
        attn_c = [None if attn_h is None else torch.empty(attn_h.shape, dtype=attn_h.dtype, device=dev)
                  for _ in range(NB)]
        masked_d = [torch.empty_like(masked) for _ in range(NB)]
        blen_h = torch.empty(B, dtype=torch.int32).pin_memory()
        plans2 = [dlm.StepPlan(dev_rows[j], dev_rows[(j - 1) % NB], masked_d[j], attn=attn_c[j], block_start=0,
                               row_index=row_index, **common) for j in range(NB)]
        outs_h = {k: torch.empty((B, blk), dtype=torch.uint8).pin_memory() for k in plans2[0].out}
        nsel_h = {k: torch.empty(B, dtype=torch.int32).pin_memory() for k in plans2[0].out}
        copy_stream = torch.cuda.Stream(device=dev)
        up_done = [torch.cuda.Event() for _ in range(NB)]
        step_done = [torch.cuda.Event() for _ in range(NB)]

        def upload(k):
            j = k % NB
            with torch.cuda.stream(copy_stream):
                if k >= 2:   # step k-2 (prev = logits set k % 3) is the set's last reader
                    copy_stream.wait_event(step_done[(k - 2) % NB])
                dev_rows[j].copy_(host_rows[j], non_blocking=True)
                if attn_c[j] is not None:
                    attn_c[j].copy_(attn_h, non_blocking=True)
                masked_d[j].copy_(masked_h, non_blocking=True)
                up_done[j].record(copy_stream)

        def decide(k):
            j = k % NB
            p = plans2[j]
            stream.wait_event(up_done[j])
            p.run(stream)
            for key in p.out:
                outs_h[key].copy_(p.out[key][0], non_blocking=True)
                nsel_h[key].copy_(p.out[key][1], non_blocking=True)
            if p.block_len is not None:
                blen_h.copy_(p.block_len, non_blocking=True)
            step_done[j].record(stream)

        def run_e2e(n):
            upload(0)
            for k in range(n):
                if k + 1 < n:
                    upload(k + 1)
                decide(k)

        run_e2e(NB + 1)                     # warm-up: every set used once
        torch.cuda.synchronize()
        a0 = torch.cuda.Event(enable_timing=True)
        a1 = torch.cuda.Event(enable_timing=True)
        a0.record(stream)
        copy_stream.wait_event(a0)
        run_e2e(args.e2e_steps)
        a1.record(stream)
        torch.cuda.synchronize()
        e2e_ms = a0.elapsed_time(a1) / args.e2e_steps
        h2d = (host_rows[0].numel() * host_rows[0].element_size() + masked_h.numel()
               + (0 if attn_h is None else attn_h.numel() * attn_h.element_size()))
        d2h = (sum(t.numel() for t in outs_h.values()) + sum(t.numel() * 4 for t in nsel_h.values())
               + (blen_h.numel() * 4 if plans2[0].block_len is not None else 0))
        e2e = {"ms_per_step": e2e_ms, "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
               "prev": "resident: the previous step's upload",
               "pipeline": "step k+1's upload (copy stream) overlaps step k's decisions; three device sets rotate"}
        if int(status.item()) != 0:
            raise RuntimeError(f"device status {int(status.item())} during the end-to-end steps")

    return dict(total_ms=total_ms, k1=k1, rules_ms=rules_ms, per_rule=per_rule, attention=attention, clocks=clocks,
                e2e=e2e, host_ms=host_ms, flush=flush, fused=list(plan.fused), folded=plan.folded,
                cfg=cfg, launches=plan.n_launches * args.steps, w=w, decisions=int(w.masked.sum()),
                rows=int(w.masked.sum()))


# ------------------------------------------------------------------ oracle
def oracle_sample(w, n_seq):
    """The oracle's whole path (statistics + the workload's rules) on the
    first n_seq sequences; returns (seconds, decisions)."""
    import oracle
    import synth

    cfg = w.cfg
    blk = cfg.blk
    rows = n_seq * blk
    cur = np.ascontiguousarray(w.cur[:rows])
    prev = np.ascontiguousarray(w.prev[:rows])
    masked = np.ascontiguousarray(w.masked[:n_seq])
    code = None if cfg.logit_dtype == synth.F32 else cfg.logit_dtype
    ri = None
    if cfg.masked_count >= 0:
        ri = np.nonzero(masked.reshape(-1))[0].astype(np.int32)
    t = time.perf_counter()
    o = oracle.row_stats(cur, prev, dtype=code, row_index=ri, n_out=rows)
    conf = o["conf"].reshape(n_seq, blk)
    if "threshold" in cfg.rules:
        oracle.select_threshold(conf, masked, cfg.tau)
    scope = None
    if "boundary" in cfg.rules:
        bl, _ = oracle.depcap_boundary(o["kl"].reshape(n_seq, blk), o["entropy"].reshape(n_seq, blk), cfg.lam,
                                       cfg.L_min)
        if cfg.name == "depcap_window":
            scope = bl
    if "cap" in cfg.rules:
        am = np.where(o["argmax"] < 0, 0, o["argmax"]).reshape(n_seq, blk)
        oracle.cap_select(cur, am, conf, o["lse"].reshape(n_seq, blk), masked, cfg.tau_low, cfg.tau_high,
                          cfg.gamma, cfg.p_max, scope_len=scope, dtype=code)
    if "dapd" in cfg.rules:
        acode = None if cfg.attn_dtype == synth.F32 else cfg.attn_dtype
        oracle.dapd(np.ascontiguousarray(w.attn[:n_seq]), masked, conf, cfg.tau_edge, cfg.bulk_conf,
                    cfg.bulk_frac, dtype=acode)
    return time.perf_counter() - t, int(masked.sum())


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo), or "unknown"."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith(("model name", "cpu part")):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


def _oracle_rate(w, budget_s):
    """Decisions per second of the oracle on repeated passes over a bounded
    sample of the workload, about ``budget_s`` seconds of work; (rate, sample)."""
    dt1, _ = oracle_sample(w, 1)
    n_seq = int(max(1, min(w.cfg.batch, budget_s / max(dt1, 1e-3))))
    total, count, reps = 0.0, 0, 0
    while total < budget_s and reps < 10000:
        dt, n = oracle_sample(w, n_seq)
        total += dt
        count += n
        reps += 1
    return count / total, (f"{reps} pass(es) of the full path (stats + four rules) over {n_seq} of "
                           f"{w.cfg.batch} sequences ({count} decisions) of the same workload, {total:.1f} s")


def cpu_baseline(w, budget_s=12.0):
    """The oracle, as it stands, on all host cores and on one thread, each
    on repeated passes over a bounded sample of the same workload."""
    import oracle
    oracle.build()
    cores = oracle.get_threads()
    value, sample = _oracle_rate(w, budget_s)
    oracle.set_threads(1)
    try:
        one, sample1 = _oracle_rate(w, budget_s / 4)
    finally:
        oracle.set_threads(cores)
    return {"value": value, "unit": "decisions/s", "cores": cores, "kind": "oracle", "sample": sample,
            "cpu_model": cpu_model(), "one_thread": {"value": one, "unit": "decisions/s", "sample": sample1}}


def run_reference(args, rank, world):
    import synth
    if rank != 0:
        return
    cfg = bench_config(args)
    w = synth.make(cfg, seed=args.seed)
    import oracle
    oracle.build()
    dt1, _ = oracle_sample(w, 1)
    per_step_budget = 150.0 / max(1, args.steps + args.warmup)
    n_seq = int(max(1, min(cfg.batch, per_step_budget / max(dt1, 1e-3))))
    for _ in range(args.warmup):
        oracle_sample(w, n_seq)
    times, n = [], 0
    for _ in range(args.steps):
        dt, n = oracle_sample(w, n_seq)
        times.append(dt)
    total = sum(times)
    value = n * args.steps / total
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "decisions/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000 * total / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": workload_desc(cfg) + f"; each step a sample of {n_seq} sequences"},
            "cpu_baseline": {"value": value, "unit": "decisions/s", "cores": oracle.get_threads(), "kind": "oracle",
                             "sample": f"{n_seq} of {cfg.batch} sequences per step", "cpu_model": cpu_model()},
            "e2e": {"value": value, "unit": "decisions/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_driver(args):
    """Whole decodes of the synthetic problem, one per rule: steps per
    sequence (NFE), wrong-token rate and the decode's device time when the
    whole decode is replayed as one CUDA graph (the stand-in model's torch
    ops included)."""
    import torch

    import synth
    from diffusion_decoding_token_gb300.driver import RULES, SyntheticDecoder
    cfg = synth.DecodeConfig(batch=args.batch or 64, blk=32, vocab=32768)
    prob = synth.decode_problem(cfg, seed=args.seed)
    dev = torch.device("cuda:0")
    out = {}
    for rule in RULES:
        dec = SyntheticDecoder(prob, rule, dev)
        dec.capture()
        times = []
        for _ in range(max(3, args.warmup) + 5):
            dec.reset()
            torch.cuda.synchronize(dev)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            dec.graph.replay()
            e1.record()
            torch.cuda.synchronize(dev)
            times.append(e0.elapsed_time(e1))
        sm = dec.summary()
        ms = statistics.median(times[max(3, args.warmup):])
        out[rule] = {"mean_steps": sm["mean_steps"], "max_steps": int(sm["steps"].max()),
                     "error_rate": sm["error_rate"], "tokens_per_step": sm["tokens_per_step"],
                     "unfinished": sm["unfinished"], "graph_steps": dec.graph_steps, "ms_per_decode": ms,
                     "tokens_per_s": cfg.batch * cfg.blk / (ms / 1000.0), "status": sm["status"]}
    # DepCap's block loop over a 256-token generation (page defaults L_max 128,
    # L_min 8, lambda 1.2; banded dependencies reach 10 positions)
    from diffusion_decoding_token_gb300.driver import DepCapDecoder
    dcfg = synth.DecodeConfig(name="depcap_loop", batch=args.batch or 64, blk=256, vocab=16384, band=10,
                              p_link=0.01)
    dprob = synth.decode_problem(dcfg, seed=args.seed)
    dec = DepCapDecoder(dprob, dev, L_max=128, L_min=8, lam=1.2)
    dec.capture()
    times = []
    for _ in range(max(3, args.warmup) + 3):
        dec.reset()
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        dec.graph.replay()
        e1.record()
        torch.cuda.synchronize(dev)
        times.append(e0.elapsed_time(e1))
    sm = dec.summary()
    ms = statistics.median(times[max(3, args.warmup):])
    out["depcap_loop"] = {"mean_steps": sm["mean_steps"], "max_steps": int(sm["steps"].max()),
                          "mean_blocks": float(sm["n_blocks"].mean()), "error_rate": sm["error_rate"],
                          "tokens_per_step": sm["tokens_per_step"], "unfinished": sm["unfinished"],
                          "graph_steps": dec.graph_steps, "ms_per_decode": ms,
                          "tokens_per_s": dcfg.batch * dcfg.blk / (ms / 1000.0), "status": sm["status"],
                          "config": {"batch": dcfg.batch, "gen_len": dcfg.blk, "vocab": dcfg.vocab, "L_max": 128,
                                     "L_min": 8, "lambda": 1.2}}
    print(json.dumps({"mode": "decode_driver", "data": "synthetic",
                      "config": {"batch": cfg.batch, "blk": cfg.blk, "vocab": cfg.vocab, "logits": "f32",
                                 "attention": f"f16 {cfg.n_layers}x{cfg.n_heads} over the block"},
                      "rules": out}), flush=True)


def main():
    args = parse()
    if args.driver:
        run_driver(args)
        return
    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as td
        td.init_process_group("nccl" if args.impl == "native" else "gloo")
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    import torch
    r = run_native(args, rank, world, local)
    cfg = r["cfg"]
    total_ms = max_over_ranks(r["total_ms"], world, f"cuda:{local}")
    if rank != 0:
        return
    value = job_throughput(r["decisions"], world, args.steps, total_ms)
    ms_step = total_ms / args.steps
    k1_ms = statistics.mean(r["k1"])
    k1_bytes = row_pass_bytes(cfg, r["w"], r["rows"], r["folded"])
    k1_gbs = k1_bytes / (k1_ms / 1000.0) / 1e9
    peak, peak_kind = load_peaks()
    line = {
        "metric": METRIC, "value": value, "unit": "decisions/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": workload_desc(cfg), "batch_per_gpu": cfg.batch, "positions_per_seq": cfg.blk,
                   "vocab": cfg.vocab,
                   "l2": (f"flushed: a 512 MB write before every timed step ({k1_bytes / 1e6:.1f} MB read by the row pass "
                          f"per step), each step timed alone" if r["flush"] else
                          f"no flush: {k1_bytes / 1e9:.3f} GB read by the row pass per step, larger than L2"),
                   "parallelism": f"dp{world}"},
        "logit_gbps": k1_gbs,
        "kernels_ms": {"row_stats": k1_ms, "row_stats_median": statistics.median(r["k1"]),
                       "rules_graph": r["rules_ms"]},
        "device": device_info(local),
        "step_structure": ("row pass on a " + ("low" if args.dapd_priority == "high" else "high") +
                           "-priority stream; DAPD attention graph on a " + args.dapd_priority +
                           "-priority side stream from the step's start (" +
                           ("after the row pass" if args.late_dapd_fork else
                            "it takes SMs from the start" if args.dapd_priority == "high" else
                            "it shares the row pass's last wave") +
                           "), DAPD selection after the row pass; threshold / boundary / CAP as " +
                           ("one chain" if args.serial_rules else "parallel branches") + "; " +
                           ("eager launches" if args.no_graph else
                            "row pass and DAPD chain launched each step, the rules replayed as a captured CUDA "
                            "graph" if not args.whole_graph else
                            "every timed step captured in CUDA graphs (250 steps per graph, the row-pass timing "
                            "events are event nodes inside them)") +
                           " (rules_graph = the rules alone, replayed as one graph, L2 warm)"),
        "host_enqueue_ms_per_step": r["host_ms"],
        "cuda_graphs": "none" if args.no_graph else ("whole steps" if args.whole_graph else "rules"),
        "roofline": {"bound": "hbm", "achieved": k1_gbs, "peak": peak, "unit": "GB/s", "frac": k1_gbs / peak,
                     "traffic": recorded_traffic() if (cfg.batch == 64 and not args.compact_attn) else None, "kernel": "row_stats", "peak_kind": peak_kind,
                     "algorithmic_bytes": k1_bytes},
        "gpu_launches": r["launches"],
        "fused_rules": r["fused"],
        "folded_attention": r["folded"],
        "per_rule": r["per_rule"],
    }
    if r["attention"]:
        a = r["attention"]
        line["attention"] = dict(a, peak=peak, frac=a["gbps"] / peak, unit="GB/s")
    if r["clocks"]:
        line["clocks"] = r["clocks"]
    if r["e2e"]:
        e = r["e2e"]
        line["e2e"] = {"value": r["decisions"] * world / (e["ms_per_step"] / 1000.0), "unit": "decisions/s",
                       "h2d_bytes_per_step": e["h2d_bytes_per_step"], "d2h_bytes_per_step": e["d2h_bytes_per_step"],
                       "ms_per_step": e["ms_per_step"], "prev": e["prev"]}
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(r["w"])
    line["config"]["workload_name"] = cfg.name
    if world == 1 and not args.no_per_workload and not args.batch and not args.compact_attn:
        del r
        line["per_workload"] = per_workload(args, cfg.name, peak, local)
    print(json.dumps(line), flush=True)


def per_workload(args, headline, peak, local):
    """Short runs of the other workloads in the same launch configuration
    (the headline's graph mode, L2 flushed before every step when the step's
    rows fit in it): ms per step, decisions/s, the row pass's GB/s against
    the peak, and the oracle's rate on the host cores."""
    import torch

    import synth
    out = {}
    for name in synth.ORDER:
        if name == headline:
            continue
        a = argparse.Namespace(**vars(args))
        a.workload, a.steps, a.warmup, a.e2e_steps = name, args.per_workload_steps, 3, 0
        a.seed = 1000 + synth.ORDER.index(name)
        r = run_native(a, 0, 1, local, light=True)
        cfg = r["cfg"]
        k1_bytes = row_pass_bytes(cfg, r["w"], r["rows"], r["folded"])
        k1_ms = statistics.mean(r["k1"])
        ms = r["total_ms"] / a.steps
        rec = {"workload": workload_desc(cfg), "steps": a.steps, "ms_per_step": ms,
               "decisions_per_s": r["decisions"] / (ms / 1000.0),
               "row_pass": {"ms": k1_ms, "gbps": k1_bytes / (k1_ms / 1000.0) / 1e9,
                            "frac": k1_bytes / (k1_ms / 1000.0) / 1e9 / peak, "algorithmic_bytes": k1_bytes},
               "l2": "flushed before every step" if r["flush"] else "not flushed (rows larger than L2)",
               "gpu_launches": r["launches"], "fused_rules": r["fused"], "folded_attention": r["folded"]}
        if not args.no_cpu_baseline:
            import oracle
            oracle.build()
            v, sample = _oracle_rate(r["w"], 2.0)
            rec["cpu_baseline"] = {"value": v, "unit": "decisions/s", "cores": oracle.get_threads(),
                                   "kind": "oracle", "sample": sample}
        out[name] = rec
        del r
        torch.cuda.empty_cache()
    return out


if __name__ == "__main__":
    main()
