"""Seeded synthetic inputs for the per-step unmask decision.

This module only draws random numbers and lays them out; it holds none of the
decision arithmetic (no softmax statistics, no selection rule), so both the
CUDA path and the CPU oracle can be fed from it without sharing code.

The workloads stand in for the pages' LLaDA / Dream decoding settings
(generation length 256, blocks of 32, vocabularies of 126464 and 152064; see
"DepCap", Experiments, and the Fast-dLLM review, Validation).  No benchmark
items are used or reproduced: every value is drawn from the recipe below.

Recipe (per sequence, independent PCG64 streams keyed by (seed, sequence,
attempt) so one sequence can be redrawn without touching the others):

* logits: background N(0, sigma^2); a fraction of the rows ("boosted") get one
  random token raised so that its softmax confidence is about sigmoid(u) with
  u ~ U(lo, hi): the token is set to u + ln(V-1) + sigma^2/2, the expected
  log-mass of the background (the "relative" reading).  ``boost_mode=
  "absolute"`` instead adds u to the token's background value (the literal
  reading).  Conflicts for CAP are planted between boosted rows i, j by
  raising z_i[tok_j] and z_j[tok_i] to 5 below the rows' own top values.
* previous-step logits: current + N(0, prev_sigma^2) (row k of the DepCap
  window uses prev_sigma * exp(-k/16) and the roles "before"/"after").
* attention block (the [blk, blk] submatrix of every layer and head):
  scores N(0, attn_sigma^2), planted links (a band plus random pairs, shared by
  all layers and heads) raised by beta = ln(4 tau Z) with Z = N e^{sigma^2/2},
  rows normalised over all N columns, the N - blk columns outside the block
  entering through their expected mass.  Stored as f16 (f32 for the tiny case).
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace
import math
import os

import numpy as np

F32, BF16, F16 = 0, 1, 2


@dataclass(frozen=True)
class Config:
    name: str
    batch: int
    blk: int                 # positions per sequence (active block or DepCap window)
    vocab: int
    logit_dtype: int
    sigma: float             # background logit std
    boost_lo: float
    boost_hi: float
    boost_frac: float        # fraction of rows given a peaked token
    prev_sigma: float
    prev_decay: float = 0.0  # >0: prev_sigma * exp(-k / prev_decay) over row k (DepCap window)
    conflict_partners: float = 2.0   # planted CAP conflicts per boosted row (mean)
    conflict_pair_cap: float = 0.10  # never more than this fraction of pairs
    # attention (n_layers == 0: none)
    n_layers: int = 0
    n_heads: int = 0
    seq_len: int = 0
    block_start: int = 0
    attn_dtype: int = F16
    attn_sigma: float = 1.0
    prompt_boost: float = 0.0
    band: int = 1
    p_link: float = 0.05
    masked_count: int = -1   # -1: every position of the block is masked
    # decision parameters
    tau: float = 0.9
    tau_edge: float = 0.01
    bulk_conf: float = 0.9
    bulk_frac: float = 0.5
    lam: float = 1.0
    L_min: int = 8
    tau_low: float = 0.8
    tau_high: float = 0.95
    gamma: float = -16.0
    p_max: int = 32
    rules: tuple = ("threshold", "boundary", "cap", "dapd")
    boost_mode: str = "relative"


CONFIGS: dict[str, Config] = {
    "tiny": Config(
        name="tiny", batch=1, blk=32, vocab=1024, logit_dtype=F32, sigma=1.0,
        boost_lo=2.0, boost_hi=8.0, boost_frac=1.0, prev_sigma=0.3,
        n_layers=2, n_heads=4, seq_len=64, block_start=32, attn_dtype=F32,
        attn_sigma=0.25, prompt_boost=1.0, band=1, p_link=0.05,
        tau_edge=0.02, L_min=4, p_max=32),
    "llada_step": Config(
        name="llada_step", batch=1, blk=32, vocab=126464, logit_dtype=BF16, sigma=2.0,
        boost_lo=4.0, boost_hi=12.0, boost_frac=0.6, prev_sigma=0.3,
        n_layers=10, n_heads=32, seq_len=512, block_start=256, p_max=32),
    "depcap_window": Config(
        name="depcap_window", batch=1, blk=64, vocab=126464, logit_dtype=BF16, sigma=2.0,
        boost_lo=4.0, boost_hi=12.0, boost_frac=0.6, prev_sigma=1.0, prev_decay=16.0,
        tau_low=0.7, tau_high=0.95, p_max=64, rules=("boundary", "cap")),
    "batched": Config(
        name="batched", batch=64, blk=32, vocab=152064, logit_dtype=BF16, sigma=2.0,
        boost_lo=4.0, boost_hi=12.0, boost_frac=0.6, prev_sigma=0.3,
        n_layers=10, n_heads=28, seq_len=512, block_start=256, p_max=32),
    "stress_graph": Config(
        name="stress_graph", batch=8, blk=256, vocab=126464, logit_dtype=BF16, sigma=2.0,
        boost_lo=4.0, boost_hi=12.0, boost_frac=0.6, prev_sigma=0.3,
        n_layers=10, n_heads=32, seq_len=1024, block_start=768, band=2, p_link=0.02,
        p_max=256),
    "stress_bulk": Config(
        name="stress_bulk", batch=8, blk=256, vocab=126464, logit_dtype=BF16, sigma=2.0,
        boost_lo=4.0, boost_hi=12.0, boost_frac=0.6, prev_sigma=0.3,
        n_layers=10, n_heads=32, seq_len=1024, block_start=768, band=2, p_link=0.02,
        masked_count=100, p_max=256, rules=("threshold", "cap", "dapd")),
}

# the pages' five workloads in order (the last one has two phases)
ORDER = ["tiny", "llada_step", "depcap_window", "batched", "stress_graph", "stress_bulk"]


def scaled(cfg: Config, **kw) -> Config:
    """A copy of ``cfg`` with some fields replaced (smaller test variants)."""
    return replace(cfg, **kw)


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bf16 (nearest, ties to even) and return the bit patterns."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def from_bf16_bits(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32)


def to_f16_bits(x: np.ndarray) -> np.ndarray:
    return np.ascontiguousarray(x, dtype=np.float32).astype(np.float16).view(np.uint16)


def _rng(seed: int, seq: int, attempt: int, stream: int) -> np.random.Generator:
    return np.random.default_rng(np.random.SeedSequence([int(seed), int(seq), int(attempt), int(stream)]))


def _store(x: np.ndarray, dtype: int) -> np.ndarray:
    if dtype == F32:
        return np.ascontiguousarray(x, dtype=np.float32)
    if dtype == BF16:
        return to_bf16_bits(x)
    return to_f16_bits(x)


def sequence_logits(cfg: Config, seed: int, seq: int, attempt: int = 0):
    """(cur, prev) logits of one sequence, [blk, V] in storage form, plus the
    planted tokens/boosts for reference."""
    rng = _rng(seed, seq, attempt, 0)
    blk, V, sg = cfg.blk, cfg.vocab, cfg.sigma
    z = rng.standard_normal((blk, V), dtype=np.float32)
    z *= np.float32(sg)
    boosted = rng.random(blk) < cfg.boost_frac
    tok = rng.integers(0, V, blk)
    u = rng.uniform(cfg.boost_lo, cfg.boost_hi, blk)
    rows = np.nonzero(boosted)[0]
    top = np.zeros(blk, np.float64)
    for i in rows:
        if cfg.boost_mode == "relative":
            top[i] = u[i] + math.log(V - 1) + sg * sg / 2.0
        else:
            top[i] = float(z[i, tok[i]]) + u[i]
        z[i, tok[i]] = top[i]
    nb = len(rows)
    if nb > 1 and cfg.conflict_partners > 0:
        p_pair = min(cfg.conflict_pair_cap, cfg.conflict_partners / (nb - 1))
        pick = rng.random((nb, nb)) < p_pair
        for a in range(nb):
            for b in range(a + 1, nb):
                if pick[a, b]:
                    i, j = rows[a], rows[b]
                    if tok[i] != tok[j]:
                        z[i, tok[j]] = top[i] - 5.0
                        z[j, tok[i]] = top[j] - 5.0
    rng_p = _rng(seed, seq, attempt, 1)
    noise = rng_p.standard_normal((blk, V), dtype=np.float32)
    if cfg.prev_decay > 0:
        scale = (cfg.prev_sigma * np.exp(-np.arange(blk) / cfg.prev_decay)).astype(np.float32)
        noise *= scale[:, None]
    else:
        noise *= np.float32(cfg.prev_sigma)
    other = z + noise
    if cfg.prev_decay > 0:
        # DepCap window: the stored "previous" row is the distribution before
        # the last block was decoded, the "current" one after it.
        cur, prev = other, z
    else:
        cur, prev = z, other
    return _store(cur, cfg.logit_dtype), _store(prev, cfg.logit_dtype), dict(
        boosted=boosted, token=tok, u=u)


def planted_links(cfg: Config, rng: np.random.Generator) -> np.ndarray:
    blk = cfg.blk
    idx = np.arange(blk)
    P = (np.abs(idx[:, None] - idx[None, :]) <= cfg.band) & (idx[:, None] != idx[None, :])
    R = rng.random((blk, blk)) < cfg.p_link
    R = np.triu(R, 1)
    P |= R | R.T
    return P


def sequence_attention(cfg: Config, seed: int, seq: int, attempt: int = 0):
    """Block submatrix [L, H, blk, blk] of one sequence's attention maps."""
    rng = _rng(seed, seq, attempt, 2)
    blk, N, sg = cfg.blk, cfg.seq_len, cfg.attn_sigma
    P = planted_links(cfg, rng)
    x = rng.standard_normal((cfg.n_layers, cfg.n_heads, blk, blk), dtype=np.float32)
    x *= np.float32(sg)
    e_half = math.exp(sg * sg / 2.0)
    if cfg.prompt_boost:
        z_rest = (N - blk) * e_half * math.exp(cfg.prompt_boost)
        z_all = z_rest + blk * e_half
    else:
        z_rest = (N - blk) * e_half
        z_all = N * e_half
    beta = math.log(4.0 * cfg.tau_edge * z_all)
    x[:, :, P] += np.float32(beta)
    w = np.exp(x.astype(np.float64))
    a = w / (w.sum(axis=-1, keepdims=True) + z_rest)
    return _store(a.astype(np.float32), cfg.attn_dtype), P


def sequence_mask(cfg: Config, seed: int, seq: int, attempt: int = 0) -> np.ndarray:
    m = np.ones(cfg.blk, np.uint8)
    if cfg.masked_count >= 0:
        rng = _rng(seed, seq, attempt, 3)
        m[:] = 0
        m[rng.choice(cfg.blk, cfg.masked_count, replace=False)] = 1
    return m


@dataclass
class Workload:
    cfg: Config
    seed: int
    cur: np.ndarray          # [B*blk, V] storage
    prev: np.ndarray
    masked: np.ndarray       # [B, blk] uint8
    attn: np.ndarray | None  # [B, L, H, blk, blk] storage (block submatrix)
    links: np.ndarray | None  # [B, blk, blk] planted links
    attempts: np.ndarray = field(default=None)

    def replace_sequence(self, b: int, attempt: int) -> None:
        """Redraw sequence ``b`` with another attempt number."""
        cfg = self.cfg
        c, p, _ = sequence_logits(cfg, self.seed, b, attempt)
        self.cur[b * cfg.blk:(b + 1) * cfg.blk] = c
        self.prev[b * cfg.blk:(b + 1) * cfg.blk] = p
        self.masked[b] = sequence_mask(cfg, self.seed, b, attempt)
        if self.attn is not None:
            a, P = sequence_attention(cfg, self.seed, b, attempt)
            self.attn[b] = a
            self.links[b] = P
        self.attempts[b] = attempt


def make(cfg: Config | str, seed: int, attempts=None) -> Workload:
    """Draw a whole workload; ``attempts[b]`` picks the stream of sequence b."""
    if isinstance(cfg, str):
        cfg = CONFIGS[cfg]
    B, blk, V = cfg.batch, cfg.blk, cfg.vocab
    att = np.zeros(B, np.int64) if attempts is None else np.asarray(attempts, np.int64).copy()
    st = np.float32 if cfg.logit_dtype == F32 else np.uint16
    cur = np.empty((B * blk, V), st)
    prev = np.empty((B * blk, V), st)
    masked = np.empty((B, blk), np.uint8)
    attn = links = None
    if cfg.n_layers:
        at = np.float32 if cfg.attn_dtype == F32 else np.uint16
        attn = np.empty((B, cfg.n_layers, cfg.n_heads, blk, blk), at)
        links = np.empty((B, blk, blk), bool)
    w = Workload(cfg, seed, cur, prev, masked, attn, links, att)
    # sequences are independent streams: draw them on a few threads (numpy
    # releases the GIL in its bulk kernels); the result does not depend on it
    from concurrent.futures import ThreadPoolExecutor
    workers = max(1, min(B, os.cpu_count() or 1, 16))
    if workers == 1:
        for b in range(B):
            w.replace_sequence(b, int(att[b]))
    else:
        with ThreadPoolExecutor(workers) as ex:
            list(ex.map(lambda b: w.replace_sequence(b, int(att[b])), range(B)))
    return w


# ---------------------------------------------------------------------------
# Multi-step decoding problems (inputs of the synthetic decode driver).
#
# Per sequence of blk positions: a planted dependency graph (band + random
# links, the same recipe as the attention), a target token t_i and a decoy
# d_i per position, background logits N(0, sigma^2), a target margin
# u_i ~ U(u_lo, u_hi) and a decoy strength v_i ~ U(0, v_hi).  The state-
# dependent logits are formed by the driver (see
# diffusion_decoding_token_gb300.driver): with s_i the fraction of i's
# neighbours already decoded,
#     z_i[t_i] = c0 + u_i + kappa * s_i,   z_i[d_i] = c0 + v_i * (1 - s_i),
# c0 = ln(V - 1) + sigma^2 / 2 (the background's expected log-mass), so a
# position whose neighbours are still masked may prefer its decoy.
# ---------------------------------------------------------------------------
@dataclass(frozen=True)
class DecodeConfig:
    name: str = "decode_small"
    batch: int = 16
    blk: int = 32
    vocab: int = 4096
    sigma: float = 1.0
    u_lo: float = 0.0
    u_hi: float = 6.0
    v_hi: float = 5.0
    kappa: float = 6.0
    band: int = 1
    p_link: float = 0.05
    n_layers: int = 2
    n_heads: int = 4
    tau_edge: float = 0.05


def decode_problem(cfg: DecodeConfig, seed: int, attempts=None) -> dict:
    """Static inputs of one multi-step decoding problem (numpy arrays);
    ``attempts[b]`` picks the stream of sequence b (default 0), so one
    sequence can be redrawn without touching the others."""
    B, blk, V = cfg.batch, cfg.blk, cfg.vocab
    att = np.zeros(B, np.int64) if attempts is None else np.asarray(attempts, np.int64)
    base = np.empty((B * blk, V), np.float32)
    target = np.empty((B, blk), np.int64)
    decoy = np.empty((B, blk), np.int64)
    u = np.empty((B, blk), np.float32)
    v = np.empty((B, blk), np.float32)
    links = np.empty((B, blk, blk), bool)
    attn = np.empty((B, cfg.n_layers, cfg.n_heads, blk, blk), np.uint16)
    acfg = Config(name="decode_attn", batch=1, blk=blk, vocab=1, logit_dtype=F32, sigma=1.0, boost_lo=0,
                  boost_hi=0, boost_frac=0, prev_sigma=0, n_layers=cfg.n_layers, n_heads=cfg.n_heads,
                  seq_len=blk, band=cfg.band, p_link=cfg.p_link, tau_edge=cfg.tau_edge, attn_sigma=0.25)
    for b in range(B):
        rng = _rng(seed, b, int(att[b]), 10)
        base[b * blk:(b + 1) * blk] = rng.standard_normal((blk, V), dtype=np.float32) * np.float32(cfg.sigma)
        t = rng.integers(0, V, blk)
        d = (t + rng.integers(1, V, blk)) % V
        target[b], decoy[b] = t, d
        u[b] = rng.uniform(cfg.u_lo, cfg.u_hi, blk).astype(np.float32)
        v[b] = rng.uniform(0.0, cfg.v_hi, blk).astype(np.float32)
        a, P = sequence_attention(acfg, seed + 7919, b, int(att[b]))
        attn[b] = a
        links[b] = P
    c0 = np.float32(math.log(V - 1) + cfg.sigma * cfg.sigma / 2.0)
    return dict(cfg=cfg, base=base, target=target, decoy=decoy, u=u, v=v, links=links, attn=attn, c0=c0,
                attempts=att.copy())
