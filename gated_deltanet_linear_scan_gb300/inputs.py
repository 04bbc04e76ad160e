"""Seeded synthetic inputs for the gated delta-rule block (shared by tests and bench).

This module only draws random numbers; it computes nothing the block computes.
Every array is float32 (int32 for slot ids), generated on the host with NumPy's
PCG64. Each array of each sequence (and each decode step) has its own
SeedSequence keyed by (1000 + config id, a tag, sequence or slot, step), so any
subset of sequences can be regenerated on its own, bit for bit.

Distributions (the workloads' recipe):
  qkv ~ N(0,1); conv weight ~ N(0, 0.5^2); conv_state ~ N(0,1);
  initial state ~ N(0, 0.1^2); gated-norm weight ~ N(1, 0.1^2); z ~ N(0,1);
  beta = sigmoid(N(0,1)) (drawn as logits b for the raw-gate block API);
  g (log-decay) ~ U(-2, -0.01), or U(-0.5, -0.001) for the long scan.
For the raw-gate block API g is reached through a = -exp(A_log) with
A_log ~ U(-0.5, 0.5), dt ~ N(0, 0.5^2) and alpha = log(expm1(g / a)) - dt, the
inverse of the gate, so the realised g has exactly the stated distribution.
For the recurrence-only API q and k are drawn uniformly on the unit sphere
(a normalised Gaussian), matching "q, k L2-normed after conv+SiLU".
"""
from dataclasses import dataclass, field, replace
from typing import Optional, Tuple

import numpy as np


@dataclass(frozen=True)
class Config:
    cid: int
    name: str
    n_seqs: int
    n_k_heads: int
    n_v_heads: int
    state_size: int
    conv_kernel: int = 4
    n_tokens: int = 1          # tokens per sequence for a scan
    steps: int = 1             # chained decode steps
    pool: Optional[int] = None  # serving pool size (None: one slot per sequence)
    g_range: Tuple[float, float] = (-2.0, -0.01)
    eps: float = 1e-6
    desc: str = field(default="", compare=False)

    @property
    def conv_dim(self):
        return 2 * self.n_k_heads * self.state_size + self.n_v_heads * self.state_size

    @property
    def key_dim(self):
        return self.n_k_heads * self.state_size

    @property
    def pool_size(self):
        return self.n_seqs if self.pool is None else self.pool

    @property
    def scale(self):
        return float(np.float32(1.0 / np.sqrt(self.state_size)))

    @property
    def seed(self):
        return 1000 + self.cid


CONFIGS = {
    0: Config(0, "tiny_oracle_check", n_seqs=1, n_k_heads=2, n_v_heads=4, state_size=32,
              n_tokens=16, steps=16, desc="N=1 Hk=2 H=4 S=32 C=256 T=16"),
    1: Config(1, "single_seq_decode_1000", n_seqs=1, n_k_heads=16, n_v_heads=32, state_size=128,
              steps=1000, desc="N=1 Hk=16 H=32 S=128 C=8192, 1000 chained decode steps"),
    2: Config(2, "prefill_scan_4x4096", n_seqs=4, n_k_heads=16, n_v_heads=32, state_size=128,
              n_tokens=4096, g_range=(-0.5, -0.001),
              desc="N=4 T=4096 Hk=16 H=32 S=128, sequential scan"),
    3: Config(3, "batched_decode_64", n_seqs=64, n_k_heads=16, n_v_heads=32, state_size=128,
              steps=200, desc="N=64 one token each, Hk=16 H=32 S=128, 200 chained steps"),
    4: Config(4, "serving_pool_256_of_512", n_seqs=256, n_k_heads=16, n_v_heads=32,
              state_size=128, steps=50, pool=512,
              desc="256 active slots of a 512-slot pool, Hk=16 H=32 S=128"),
}


def get_config(which, **overrides):
    """One of the five workloads, optionally with fields replaced (a new `cid`
    gives the variant its own seeds)."""
    cfg = CONFIGS[which]
    return replace(cfg, **overrides) if overrides else cfg


_TAGS = {"state": 1, "conv_state": 2, "conv_w": 3, "norm_w": 4, "gate_params": 5, "slots": 6,
         "qkv": 11, "gate": 12, "b": 13, "z": 14, "q": 21, "k": 22, "v": 23, "g": 24, "beta": 25,
         "pqkv": 31, "pgate": 32, "pb": 33, "pz": 34, "lengths": 41}


def _rng(cfg, tag, idx=0, step=0):
    return np.random.Generator(np.random.PCG64(
        np.random.SeedSequence([cfg.seed, _TAGS[tag], int(idx), int(step)])))


def _normal(rng, shape, std=1.0, mean=0.0):
    x = rng.standard_normal(shape, dtype=np.float32)
    if std != 1.0:
        x *= np.float32(std)
    if mean != 0.0:
        x += np.float32(mean)
    return x


def _uniform(rng, lo, hi, shape):
    return (rng.random(shape, dtype=np.float32) * np.float32(hi - lo) + np.float32(lo))


# ---- per-slot / shared parameters -----------------------------------------------------

def slots(cfg):
    """int32 slot ids of the active sequences (None when there is no pool)."""
    if cfg.pool is None:
        return None
    perm = _rng(cfg, "slots").permutation(cfg.pool)
    return perm[: cfg.n_seqs].astype(np.int32)


def state_slot(cfg, slot):
    """Initial recurrent state of one pool slot, [H][S][S] ~ N(0, 0.1^2)."""
    H, S = cfg.n_v_heads, cfg.state_size
    return _normal(_rng(cfg, "state", slot), (H, S, S), std=0.1)


def state_pool(cfg, which=None):
    """Initial state for every pool slot (or the listed slots), [P][H][S][S]."""
    ids = range(cfg.pool_size) if which is None else which
    return np.stack([state_slot(cfg, s) for s in ids])


def conv_state_slot(cfg, slot):
    return _normal(_rng(cfg, "conv_state", slot), (cfg.conv_dim, cfg.conv_kernel - 1))


def conv_state_pool(cfg, which=None):
    ids = range(cfg.pool_size) if which is None else which
    return np.stack([conv_state_slot(cfg, s) for s in ids])


def conv_weight(cfg):
    return _normal(_rng(cfg, "conv_w"), (cfg.conv_dim, cfg.conv_kernel), std=0.5)


def norm_weight(cfg):
    return _normal(_rng(cfg, "norm_w"), (cfg.state_size,), std=0.1, mean=1.0)


def gate_params(cfg):
    """(dt [H], a [H]) with a = -exp(A_log), A_log ~ U(-0.5, 0.5), dt ~ N(0, 0.5^2)."""
    rng = _rng(cfg, "gate_params")
    H = cfg.n_v_heads
    a_log = rng.uniform(-0.5, 0.5, H)
    dt = rng.standard_normal(H) * 0.5
    return dt.astype(np.float32), (-np.exp(a_log)).astype(np.float32)


# ---- per-step activations of the raw-gate block ---------------------------------------

def block_step(cfg, step, seqs=None):
    """Per-sequence inputs of one decode step of the block.

    Returns dict qkv [n][C], alpha [n][H], b [n][H], z [n][H][S] for the listed
    sequence indices (all by default)."""
    seqs = range(cfg.n_seqs) if seqs is None else seqs
    dt, a = gate_params(cfg)
    H, S, C = cfg.n_v_heads, cfg.state_size, cfg.conv_dim
    lo, hi = cfg.g_range
    qkv, alpha, b, z = [], [], [], []
    for n in seqs:
        qkv.append(_normal(_rng(cfg, "qkv", n, step), (C,)))
        g = _rng(cfg, "gate", n, step).uniform(lo, hi, H)
        alpha.append((np.log(np.expm1(g / a.astype(np.float64))) - dt).astype(np.float32))
        b.append(_normal(_rng(cfg, "b", n, step), (H,)))
        z.append(_normal(_rng(cfg, "z", n, step), (H, S)))
    return {"qkv": np.stack(qkv), "alpha": np.stack(alpha), "b": np.stack(b),
            "z": np.stack(z)}


def prefill_seq(cfg, n, n_tokens=None):
    """Raw block inputs of sequence n over n_tokens positions, each array drawn from
    its own stream (distributions as block_step): qkv [T][C], alpha, b [T][H],
    z [T][H][S]."""
    T = cfg.n_tokens if n_tokens is None else n_tokens
    dt, a = gate_params(cfg)
    H, S, C = cfg.n_v_heads, cfg.state_size, cfg.conv_dim
    lo, hi = cfg.g_range
    g = _uniform(_rng(cfg, "pgate", n), lo, hi, (T, H)).astype(np.float64)
    alpha = (np.log(np.expm1(g / a.astype(np.float64))) - dt).astype(np.float32)
    return {"qkv": _normal(_rng(cfg, "pqkv", n), (T, C)), "alpha": alpha,
            "b": _normal(_rng(cfg, "pb", n), (T, H)), "z": _normal(_rng(cfg, "pz", n), (T, H, S))}


def ragged_lengths(cfg, total_tokens, lo=1, hi=4096):
    """Sequence lengths of a ragged prefill batch: log-uniform in [lo, hi] (seeded), drawn
    until they add up to total_tokens (the last one trimmed to fit), so short prompts
    and long ones share a call as they do in a serving prefill batch."""
    rng = _rng(cfg, "lengths")
    lengths, left = [], int(total_tokens)
    while left > 0:
        L = int(np.exp(rng.uniform(np.log(lo), np.log(hi + 1))))
        L = min(max(L, lo), hi, left)
        lengths.append(L)
        left -= L
    return lengths


def block_static(cfg):
    dt, a = gate_params(cfg)
    return {"conv_w": conv_weight(cfg), "dt": dt, "a": a, "norm_w": norm_weight(cfg)}


# ---- recurrence-only activations (post-norm q/k, post-sigmoid beta, g) -----------------

def _unit(rng, shape):
    x = rng.standard_normal(shape, dtype=np.float32)
    x /= np.sqrt(np.einsum("...i,...i->...", x, x))[..., None]
    return x


def recurrence_seq(cfg, n, n_tokens=None):
    """q,k [T][Hk][S] (unit), v [T][H][S], g [T][H], beta [T][H] of sequence n.

    Each array of sequence n is drawn from its own stream in token order, so a
    sequence can be regenerated alone and a shorter T is a prefix of a longer one."""
    T = cfg.n_tokens if n_tokens is None else n_tokens
    Hk, H, S = cfg.n_k_heads, cfg.n_v_heads, cfg.state_size
    lo, hi = cfg.g_range
    logit = _rng(cfg, "beta", n).standard_normal((T, H), dtype=np.float32)
    return {
        "q": _unit(_rng(cfg, "q", n), (T, Hk, S)),
        "k": _unit(_rng(cfg, "k", n), (T, Hk, S)),
        "v": _normal(_rng(cfg, "v", n), (T, H, S)),
        "g": _uniform(_rng(cfg, "g", n), lo, hi, (T, H)),
        "beta": (np.float32(1) / (np.float32(1) + np.exp(-logit))).astype(np.float32),
    }


def recurrence_batch(cfg, seqs=None, n_tokens=None):
    """Stacked recurrence_seq over sequences: q,k [N][T][Hk][S], v [N][T][H][S], ..."""
    seqs = range(cfg.n_seqs) if seqs is None else seqs
    per = [recurrence_seq(cfg, n, n_tokens) for n in seqs]
    return {key: np.stack([p[key] for p in per]) for key in per[0]}
