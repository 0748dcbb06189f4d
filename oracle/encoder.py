"""Float path of the oracle: the encoder written out step by step in fp64.

Test infrastructure only (see the package docstring).  Each function cites
the passage of the tensai page "テキスト埋め込み" that it follows; where the
page is silent the plainest reading is taken and stated in the docstring.
"""
from __future__ import annotations

import math

import numpy as np
from scipy.special import erf

from .precision import round_to_bf16


# --------------------------------------------------------------------------
# Building blocks
# --------------------------------------------------------------------------

def layernorm(x, gamma, eps: float) -> np.ndarray:
    """Bias-free LayerNorm over the last axis.

    §何が動くか / エンコーダ names a LayerNorm without bias.  Reading: the
    usual normalisation with the biased variance (divide by H), the epsilon
    inside the square root, and a learned gain only:
    y = (x - mean) / sqrt(var + eps) * gamma.
    """
    x = np.asarray(x, dtype=np.float64)
    mean = x.mean(axis=-1, keepdims=True)
    var = ((x - mean) ** 2).mean(axis=-1, keepdims=True)
    return (x - mean) / np.sqrt(var + eps) * np.asarray(gamma, dtype=np.float64)


def rope_cos_sin(positions, head_dim: int, base: float):
    """cos and sin of the rotary angles pos * base**(-2j/d), j < d/2.

    §何が動くか / エンコーダ gives RoPE with base 160000 (global layers) and
    10000 (window layers); the frequency ladder is the standard one.
    Returns two fp64 arrays of shape [len(positions), d/2].
    """
    half = head_dim // 2
    j = np.arange(half, dtype=np.float64)
    inv_freq = np.power(float(base), -2.0 * j / head_dim)
    ang = np.asarray(positions, dtype=np.float64)[:, None] * inv_freq[None, :]
    return np.cos(ang), np.sin(ang)


def apply_rope(x, positions, base: float) -> np.ndarray:
    """Rotate q or k ([L, heads, d]) by their positions.

    Reading of the pairing (the page does not fix it): "rotate half", i.e.
    dimension j is paired with j + d/2:
      x'_j       = x_j cos - x_{j+d/2} sin
      x'_{j+d/2} = x_{j+d/2} cos + x_j sin.
    """
    x = np.asarray(x, dtype=np.float64)
    half = x.shape[-1] // 2
    cos, sin = rope_cos_sin(positions, x.shape[-1], base)
    cos = cos[:, None, :]
    sin = sin[:, None, :]
    lo, hi = x[..., :half], x[..., half:]
    return np.concatenate([lo * cos - hi * sin, hi * cos + lo * sin], axis=-1)


def attention_text(q, k, v, is_global: bool, window: int, q_chunk: int = 256) -> np.ndarray:
    """Bidirectional multi-head attention inside one text.

    §何が動くか / エンコーダ: global layers see the whole text; the others
    see 64 tokens before and after.  Reading: query i may attend to key j
    iff the layer is global or |i - j| <= window (inclusive, so up to
    2*window + 1 keys).  Scores are q.k / sqrt(d); softmax subtracts the row
    maximum.  q, k, v: [L, heads, d] fp64.  Returns [L, heads, d].

    Queries are processed in chunks only to bound memory on long texts; each
    chunk computes exactly the definition.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    L, nh, d = q.shape
    scale = 1.0 / math.sqrt(d)
    out = np.empty_like(q)
    for q0 in range(0, L, q_chunk):
        q1 = min(L, q0 + q_chunk)
        if is_global:
            k0, k1 = 0, L
        else:
            k0, k1 = max(0, q0 - window), min(L, q1 - 1 + window + 1)
        if not is_global:
            qi = np.arange(q0, q1)[:, None]
            kj = np.arange(k0, k1)[None, :]
            allowed = np.abs(qi - kj) <= window
        for h in range(nh):
            s = (q[q0:q1, h, :] @ k[k0:k1, h, :].T) * scale
            if not is_global:
                s = np.where(allowed, s, -np.inf)
            s = s - s.max(axis=-1, keepdims=True)
            p = np.exp(s)
            p /= p.sum(axis=-1, keepdims=True)
            out[q0:q1, h, :] = p @ v[k0:k1, h, :]
    return out


def gelu(a) -> np.ndarray:
    """GELU with the exact Gaussian CDF: a * Phi(a) = 0.5 a (1 + erf(a / sqrt 2)).

    The page says "GeGLU" only; the erf form is the plainest reading.
    """
    a = np.asarray(a, dtype=np.float64)
    return 0.5 * a * (1.0 + erf(a / math.sqrt(2.0)))


def geglu(u, intermediate: int) -> np.ndarray:
    """GeGLU gate: the first I columns go through GELU, the second I gate them.

    Reading of "GeGLU のフィードフォワード" (§何が動くか / エンコーダ): for
    u = x Wi^T of width 2I, z = GELU(u[:, :I]) * u[:, I:].
    """
    u = np.asarray(u, dtype=np.float64)
    return gelu(u[:, :intermediate]) * u[:, intermediate:]


def pool_l2(states) -> np.ndarray:
    """Mean over every token of the text, then scale to unit length.

    §何が動くか / プーリング.  Reading: all tokens count, including the BOS
    and EOS wrappers; the norm is floored at 1e-12 so a zero mean stays zero.
    """
    s = np.asarray(states, dtype=np.float64)
    v = s.mean(axis=0)
    return v / max(float(np.linalg.norm(v)), 1e-12)


def layer_is_global(layer: int, shape) -> bool:
    """The first layer and every `global_every`-th layer after it are global."""
    return layer % shape.global_every == 0


# --------------------------------------------------------------------------
# The encoder
# --------------------------------------------------------------------------

class OracleModel:
    """Weights widened to fp64 for one storage variant.

    variant "fp32": the fp32 weights as given.
    variant "bf16": every weight (embedding, LayerNorm gains and the four
                    projections) rounded to bfloat16 first, then widened.
    variant "w8a8": projections go through the integer procedure of
                    ``oracle.w8a8``; embedding and gains stay fp32.
    variant "w4a8": the same with 4-bit weight blocks (codes in [-7, 7]).
    variant "w6a8": the same with 6-bit weight blocks (codes in [-31, 31]).

    ``weights`` needs attributes tok_emb, ln_attn, wqkv, wo, ln_mlp, wi,
    wo_ffn (lists per layer), in the layouts documented by the C header, and
    ln_emb / ln_final / w_proj when the shape enables the optional embedding
    norm, final norm or per-token projection (stored like the other gains and
    projections of the variant).
    """

    def __init__(self, weights, shape, variant: str = "fp32"):
        if variant not in ("fp32", "bf16", "w8a8", "w4a8", "w6a8"):
            raise ValueError(variant)
        self.shape = shape
        self.variant = variant
        conv = round_to_bf16 if variant == "bf16" else (lambda a: np.asarray(a, np.float32))
        wide = lambda a: conv(a).astype(np.float64)  # noqa: E731
        self.tok_emb = conv(weights.tok_emb)  # kept fp32-sized; rows are widened on use
        self.ln_attn = [wide(g) for g in weights.ln_attn]
        self.ln_mlp = [wide(g) for g in weights.ln_mlp]
        self.ln_emb = wide(weights.ln_emb) if getattr(shape, "emb_norm", False) else None
        self.ln_final = wide(weights.ln_final) if getattr(shape, "final_norm", False) else None
        names = ("wqkv", "wo", "wi", "wo_ffn")
        proj = [weights.w_proj] if getattr(shape, "proj_dim", 0) else []
        if variant in ("w8a8", "w4a8", "w6a8"):
            from .w8a8 import quantize_weight_blocks, quantize_weight_blocks4, quantize_weight_blocks6
            quant = {"w8a8": quantize_weight_blocks, "w4a8": quantize_weight_blocks4,
                     "w6a8": quantize_weight_blocks6}[variant]
            self.q = {name: [quant(np.asarray(w, np.float32)) for w in getattr(weights, name)] for name in names}
            self.q["w_proj"] = [quant(np.asarray(w, np.float32)) for w in proj]
        else:
            self.lin = {name: [wide(w) for w in getattr(weights, name)] for name in names}
            self.lin["w_proj"] = [wide(w) for w in proj]

    def linear(self, name: str, layer: int, x) -> np.ndarray:
        """y = x W^T (no bias: the page mentions none on any projection)."""
        if self.variant in ("w8a8", "w4a8", "w6a8"):
            from .w8a8 import w8a8_linear
            qw, d = self.q[name][layer]
            return w8a8_linear(x, qw, d)
        return np.asarray(x, dtype=np.float64) @ self.lin[name][layer].T


def encode_text_states(ids, model: OracleModel) -> np.ndarray:
    """Final per-token states [L, H] of one text (ids already wrapped).

    §何が動くか / エンコーダ.  Reading of the block order: pre-norm residual
    blocks,
        x += Wo . Attn(RoPE(LN_attn(x) Wqkv^T))
        x += Wo_ffn . GeGLU(LN_mlp(x) Wi^T)
    with no embedding norm and no final norm (the page names neither; pooling
    is over the final layer's output).  Positions count from 0 at the text's
    first token (BOS).  Optionally (``shape.emb_norm`` / ``shape.final_norm``,
    the published ModernBERT layout) a bias-free LayerNorm is applied to the
    token embeddings before layer 0 and to the last layer's output.
    """
    shape = model.shape
    H, nh, d, I = shape.hidden, shape.n_heads, shape.head_dim, shape.intermediate
    ids = np.asarray(ids, dtype=np.int64)
    L = ids.shape[0]
    pos = np.arange(L)
    x = model.tok_emb[ids].astype(np.float64)
    if model.ln_emb is not None:
        x = layernorm(x, model.ln_emb, shape.ln_eps)
    for l in range(shape.n_layers):
        is_global = layer_is_global(l, shape)
        base = shape.rope_base_global if is_global else shape.rope_base_local
        n = layernorm(x, model.ln_attn[l], shape.ln_eps)
        qkv = model.linear("wqkv", l, n)
        q = qkv[:, 0:H].reshape(L, nh, d)
        k = qkv[:, H:2 * H].reshape(L, nh, d)
        v = qkv[:, 2 * H:3 * H].reshape(L, nh, d)
        q = apply_rope(q, pos, base)
        k = apply_rope(k, pos, base)
        o = attention_text(q, k, v, is_global, shape.window).reshape(L, H)
        x = x + model.linear("wo", l, o)
        n = layernorm(x, model.ln_mlp[l], shape.ln_eps)
        u = model.linear("wi", l, n)
        x = x + model.linear("wo_ffn", l, geglu(u, I))
    if model.ln_final is not None:
        x = layernorm(x, model.ln_final, shape.ln_eps)
    return x


def encode_text_tokens(ids, model: OracleModel) -> np.ndarray:
    """Per-token unit vectors [L, D] of one text (multi-vector output).

    Page "Les Embeddings multimodaux dans Llama.cpp et GGUF", section
    "Problèmes restants": multi-vector embeddings come from a single linear
    layer applied to the token states.  Reading: the final per-token states
    (after the optional final norm), times the projection W_proj^T when the
    shape has one (D = proj_dim, else D = H), each scaled to unit length with
    the norm floored at 1e-12, as the pooled vector is.
    """
    s = encode_text_states(ids, model)
    if model.shape.proj_dim:
        s = model.linear("w_proj", 0, s)
    norms = np.maximum(np.linalg.norm(s, axis=1, keepdims=True), 1e-12)
    return s / norms


def encode_text(ids, model: OracleModel) -> np.ndarray:
    """Unit-norm embedding [H] of one text."""
    return pool_l2(encode_text_states(ids, model))


def encode_packed(ids, cu_seqlens, model: OracleModel, texts=None) -> np.ndarray:
    """Embeddings [n, H] of a packed batch.

    The packing paragraph of §何が動くか states that positions restart per
    text and attention stays inside each text, so a packed batch is encoded
    exactly as its texts one at a time; the oracle does precisely that.
    ``texts`` optionally restricts the work to a subset of text indices
    (rows of the result for other texts are left as NaN).
    """
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    n = cu.shape[0] - 1
    out = np.full((n, model.shape.hidden), np.nan)
    for j in (range(n) if texts is None else texts):
        out[j] = encode_text(np.asarray(ids)[cu[j]:cu[j + 1]], model)
    return out


def encode_packed_tokens(ids, cu_seqlens, model: OracleModel, texts=None) -> np.ndarray:
    """Per-token unit vectors [T, D] of a packed batch, text by text (rows of
    texts outside ``texts`` are left as NaN)."""
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    n = cu.shape[0] - 1
    width = model.shape.proj_dim or model.shape.hidden
    out = np.full((int(cu[-1]), width), np.nan)
    for j in (range(n) if texts is None else texts):
        out[cu[j]:cu[j + 1]] = encode_text_tokens(np.asarray(ids)[cu[j]:cu[j + 1]], model)
    return out
