"""Seeded synthetic inputs for the packed-varlen embedding encoder.

This module draws random numbers and nothing else: encoder shapes, weights
and packed batches of token ids.  None of the encoder's arithmetic lives
here, so both the CUDA path (tests, bench) and the CPU oracle's tests take
their inputs from it without sharing any computation.

Recipe (stated once, used everywhere):

* weights: one ``numpy.random.Generator(PCG64(seed))`` per model, drawn in a
  fixed order -- the token embedding E, then per layer gamma_attn, Wqkv, Wo,
  gamma_mlp, Wi, Wo_ffn, then (when the shape enables them) gamma_emb,
  gamma_final and the per-token projection.  Linear and embedding entries are
  N(0, 0.02^2) in fp32; LayerNorm gains are 1 + 0.02 * N(0, 1).
* outlier variant: a fixed set of hidden channels (a seeded permutation) has
  both LayerNorm gains of every layer multiplied by 20, so the inputs of the
  QKV and Wi projections carry large per-channel outliers.
* texts: each text is ``[BOS] + ids + [EOS]`` with ids uniform in
  [3, vocab); its length counts the two wrapper tokens.
* throughput sweep: lengths floor(exp(U[ln 8, ln 1025))) drawn until the
  token budget is filled exactly; seed = 1000 * size_index + batch_index.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, asdict

import numpy as np

BOS_ID = 1
EOS_ID = 2
FIRST_REGULAR_ID = 3


@dataclass(frozen=True)
class Shape:
    """Hyper-parameters of a ModernBERT-style encoder."""

    n_layers: int
    hidden: int
    n_heads: int
    head_dim: int
    intermediate: int
    vocab: int
    global_every: int = 3
    window: int = 64
    rope_base_global: float = 160000.0
    rope_base_local: float = 10000.0
    ln_eps: float = 1e-5
    # optional parts (off in the page's encoder): a LayerNorm on the token
    # embeddings, one on the last layer's output, and the width of a per-token
    # output projection (0 = none)
    emb_norm: bool = False
    final_norm: bool = False
    proj_dim: int = 0

    def as_dict(self):
        return asdict(self)


# 3 layers (layer 0 global), hidden 256, 4 heads of 64, GeGLU width 512.
TINY = Shape(n_layers=3, hidden=256, n_heads=4, head_dim=64, intermediate=512, vocab=4096)
# The Ruri-v3-310m shape: 25 layers, hidden 768, 12 heads of 64, GeGLU width 3072.
RURI_310M = Shape(n_layers=25, hidden=768, n_heads=12, head_dim=64, intermediate=3072, vocab=102400)

TINY_LENGTHS = (8, 37, 64, 150)                      # 259 tokens
ACCURACY_LENGTHS = (8, 24, 57, 110, 190, 280, 382)   # 1051 tokens
SWEEP_BUDGETS = (2048, 8192, 32768)
SWEEP_BATCHES = 20
LONG_DOC_LENGTHS = (8192,) * 8                       # 65536 tokens
OUTLIER_FRACTION = 0.05
OUTLIER_SCALE = 20.0


@dataclass
class Weights:
    """fp32 host weights, row-major, in the layout the C-ABI takes.

    wqkv[l]  : [3H, H]  rows 0..H-1 = q (head-major), H..2H-1 = k, 2H..3H-1 = v
    wo[l]    : [H, H]   input columns = concatenated heads
    wi[l]    : [2I, H]  rows 0..I-1 = GELU input a, rows I..2I-1 = gate g
    wo_ffn[l]: [H, I]
    """

    tok_emb: np.ndarray
    ln_attn: list = field(default_factory=list)
    wqkv: list = field(default_factory=list)
    wo: list = field(default_factory=list)
    ln_mlp: list = field(default_factory=list)
    wi: list = field(default_factory=list)
    wo_ffn: list = field(default_factory=list)
    ln_emb: np.ndarray | None = None      # [H], with Shape.emb_norm
    ln_final: np.ndarray | None = None    # [H], with Shape.final_norm
    w_proj: np.ndarray | None = None      # [proj_dim, H], with Shape.proj_dim > 0


def _normal(rng, shape, std):
    return rng.standard_normal(shape, dtype=np.float32) * np.float32(std)


def outlier_channels(hidden: int, seed: int = 0, fraction: float = OUTLIER_FRACTION) -> np.ndarray:
    """Seeded choice of round(fraction * hidden) hidden channels."""
    rng = np.random.Generator(np.random.PCG64(seed))
    count = int(round(fraction * hidden))
    return np.sort(rng.permutation(hidden)[:count]).astype(np.int64)


def make_weights(shape: Shape, seed: int = 0, std: float = 0.02, outliers: bool = False) -> Weights:
    """Draw a full set of fp32 weights for ``shape``."""
    H, I, L, V = shape.hidden, shape.intermediate, shape.n_layers, shape.vocab
    rng = np.random.Generator(np.random.PCG64(seed))
    w = Weights(tok_emb=_normal(rng, (V, H), std))
    for _ in range(L):
        w.ln_attn.append(np.float32(1.0) + _normal(rng, (H,), 0.02))
        w.wqkv.append(_normal(rng, (3 * H, H), std))
        w.wo.append(_normal(rng, (H, H), std))
        w.ln_mlp.append(np.float32(1.0) + _normal(rng, (H,), 0.02))
        w.wi.append(_normal(rng, (2 * I, H), std))
        w.wo_ffn.append(_normal(rng, (H, I), std))
    # the optional parts are drawn after every layer, so enabling them leaves
    # the draws above unchanged
    if shape.emb_norm:
        w.ln_emb = np.float32(1.0) + _normal(rng, (H,), 0.02)
    if shape.final_norm:
        w.ln_final = np.float32(1.0) + _normal(rng, (H,), 0.02)
    if shape.proj_dim:
        w.w_proj = _normal(rng, (shape.proj_dim, H), std)
    if outliers:
        ch = outlier_channels(H)
        for l in range(L):
            w.ln_attn[l][ch] *= np.float32(OUTLIER_SCALE)
            w.ln_mlp[l][ch] *= np.float32(OUTLIER_SCALE)
    return w


def make_batch(lengths, vocab: int, seed: int, wrap: bool = True):
    """Pack texts of the given lengths.

    Returns ``(ids int32[T], cu_seqlens int32[n+1])``.  With ``wrap`` each
    text of length >= 2 is BOS, uniform ids, EOS; a text of length 1 is a
    single uniform id.
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    parts = []
    for n in lengths:
        n = int(n)
        if n < 1:
            raise ValueError("text lengths must be >= 1")
        if wrap and n >= 2:
            body = rng.integers(FIRST_REGULAR_ID, vocab, size=n - 2, dtype=np.int64)
            parts.append(np.concatenate([[BOS_ID], body, [EOS_ID]]))
        else:
            parts.append(rng.integers(FIRST_REGULAR_ID, vocab, size=n, dtype=np.int64))
    ids = np.concatenate(parts).astype(np.int32) if parts else np.zeros(0, np.int32)
    cu = np.zeros(len(lengths) + 1, dtype=np.int32)
    cu[1:] = np.cumsum([int(n) for n in lengths])
    return ids, cu


def sweep_lengths(budget: int, rng, lo: int = 8, hi: int = 1024):
    """Log-uniform text lengths in [lo, hi], filled greedily to exactly ``budget`` tokens."""
    out = []
    remaining = budget
    while remaining >= 2:
        n = int(math.floor(math.exp(rng.uniform(math.log(lo), math.log(hi + 1)))))
        n = max(2, min(n, remaining))
        if remaining - n == 1:
            n += 1
        out.append(n)
        remaining -= n
    return out


def sweep_batch(budget: int, batch_index: int, vocab: int):
    """One batch of the throughput sweep (budgets 2048 / 8192 / 32768)."""
    size_index = SWEEP_BUDGETS.index(budget) if budget in SWEEP_BUDGETS else budget
    seed = 1000 * size_index + batch_index
    rng = np.random.Generator(np.random.PCG64(seed))
    lengths = sweep_lengths(budget, rng)
    return make_batch(lengths, vocab, seed=seed + 500_000)


def lengths_of(cu) -> list:
    cu = np.asarray(cu)
    return [int(b - a) for a, b in zip(cu[:-1], cu[1:])]
