"""Pins for the CPU oracle: each function checked against something other than itself.

The pins are brute force on tiny inputs (a scalar, loop-by-loop encoder over
the packed sequence with an explicit dense mask), closed forms (complex
rotation for RoPE, uniform-score attention, zeroed projections, single-token
texts), textbook values (the normal CDF inside GELU), library routines
(torch's bfloat16 conversion) and the page's invariants (unit norm, packing,
window vs. global on short texts).
"""
import cmath
import math
import os

import numpy as np
import pytest

import oracle
from oracle import encoder as enc
from text_embedding_encoder_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# --------------------------------------------------------------------------
# bf16 storage rounding
# --------------------------------------------------------------------------

def test_bf16_rounding_matches_torch():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(5)
    x = np.concatenate([
        rng.standard_normal(10000).astype(np.float32) * np.float32(0.02),
        rng.standard_normal(1000).astype(np.float32) * np.float32(1e4),
        # exact ties: 1 + 2^-8 rounds down to 1 (even), 1 + 3*2^-8 up to 1 + 2^-6
        np.array([1 + 2 ** -8, 1 + 3 * 2 ** -8, -(1 + 2 ** -8), 0.0, -0.0, 65504.0], np.float32),
    ])
    ours = oracle.round_to_bf16(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float32).numpy()
    assert np.array_equal(ours.view(np.uint32), ref.view(np.uint32))
    assert ours[-6] == 1.0 and ours[-5] == np.float32(1 + 2 ** -6)


# --------------------------------------------------------------------------
# LayerNorm
# --------------------------------------------------------------------------

def test_layernorm_moments_and_gain():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((17, 96)) * 3.0 + 5.0
    y = oracle.layernorm(x, np.ones(96), 0.0)
    np.testing.assert_allclose(y.mean(axis=1), 0.0, atol=1e-12)
    np.testing.assert_allclose((y ** 2).mean(axis=1), 1.0, atol=1e-12)   # biased variance
    g = rng.standard_normal(96)
    np.testing.assert_allclose(oracle.layernorm(x, g, 0.0), y * g, atol=1e-12)
    # shift and scale invariance, and eps inside the square root
    np.testing.assert_allclose(oracle.layernorm(2.5 * x - 7.0, g, 0.0), y * g, atol=1e-11)
    row = np.array([[1.0, -1.0]])     # mean 0, biased variance 1
    np.testing.assert_allclose(oracle.layernorm(row, np.ones(2), 3.0), row / 2.0)


# --------------------------------------------------------------------------
# RoPE
# --------------------------------------------------------------------------

def test_rope_identity_at_zero_and_complex_rotation():
    rng = np.random.default_rng(2)
    d, base = 64, 160000.0
    x = rng.standard_normal((5, 3, d))
    pos = np.array([0, 1, 7, 100, 8191])
    y = oracle.apply_rope(x, pos, base)
    np.testing.assert_allclose(y[0], x[0], atol=0)
    # closed form: pair (j, j + d/2) is the complex number x_j + i x_{j+d/2},
    # multiplied by exp(i * pos * base^(-2j/d))
    for t in range(5):
        for h in range(3):
            for j in range(d // 2):
                z = complex(x[t, h, j], x[t, h, j + d // 2])
                z *= cmath.exp(1j * pos[t] * base ** (-2.0 * j / d))
                assert abs(y[t, h, j] - z.real) < 1e-9
                assert abs(y[t, h, j + d // 2] - z.imag) < 1e-9


def test_rope_scores_depend_on_relative_position_only():
    rng = np.random.default_rng(3)
    q = rng.standard_normal((1, 1, 64))
    k = rng.standard_normal((1, 1, 64))
    for base in (10000.0, 160000.0):
        ref = None
        for i0 in (0, 5, 300, 4000):
            qi = oracle.apply_rope(q, np.array([i0 + 9]), base)
            kj = oracle.apply_rope(k, np.array([i0 + 2]), base)
            s = float((qi * kj).sum())
            ref = s if ref is None else ref
            assert abs(s - ref) < 1e-9
        # rotation preserves length
        r = oracle.apply_rope(q, np.array([123]), base)
        assert abs(np.linalg.norm(r) - np.linalg.norm(q)) < 1e-12


# --------------------------------------------------------------------------
# GELU / GeGLU
# --------------------------------------------------------------------------

def _normal_cdf_table():
    rows = []
    with open(os.path.join(GOLDEN, "normal_cdf.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                a, b = line.split()
                rows.append((float(a), float(b)))
    return rows


def test_gelu_against_normal_cdf_table():
    for x, phi in _normal_cdf_table():
        assert abs(float(oracle.gelu(x)) - x * phi) < 1e-14
        assert abs(float(oracle.gelu(-x)) - (-x) * (1.0 - phi)) < 1e-14
    xs = np.linspace(-6, 6, 101)
    np.testing.assert_allclose(oracle.gelu(xs) - oracle.gelu(-xs), xs, atol=1e-14)


def test_geglu_gates_the_second_half():
    a = np.array([[1.0, -0.5, 2.0]])
    g = np.array([[2.0, 4.0, 0.0]])
    u = np.concatenate([a, g], axis=1)
    phi1 = dict(_normal_cdf_table())[1.0]
    z = oracle.geglu(u, 3)
    assert abs(z[0, 0] - 2.0 * 1.0 * phi1) < 1e-14
    assert z[0, 2] == 0.0
    # swapping the halves changes the result: the first half is the GELU input
    assert not np.allclose(oracle.geglu(np.concatenate([g, a], axis=1), 3), z)


# --------------------------------------------------------------------------
# Attention
# --------------------------------------------------------------------------

def _dense_mask(lengths, window, is_global):
    """Explicit T x T mask over the packed sequence, from the definition."""
    text, pos = [], []
    for j, n in enumerate(lengths):
        for p in range(n):
            text.append(j)
            pos.append(p)
    T = len(text)
    m = np.zeros((T, T), dtype=bool)
    for i in range(T):
        for k in range(T):
            m[i, k] = text[i] == text[k] and (is_global or abs(pos[i] - pos[k]) <= window)
    return m


def _dense_attention(q, k, v, mask):
    T, nh, d = q.shape
    out = np.zeros_like(q)
    for h in range(nh):
        for i in range(T):
            keys = np.nonzero(mask[i])[0]
            s = np.array([q[i, h] @ k[j, h] for j in keys]) / math.sqrt(d)
            w = np.exp(s - s.max())
            w /= w.sum()
            out[i, h] = (w[:, None] * v[keys, h]).sum(axis=0)
    return out


@pytest.mark.parametrize("lengths", [[1, 2, 3], [64, 65, 66], [129, 130], [40], [7, 1, 33]])
@pytest.mark.parametrize("is_global", [True, False])
def test_attention_matches_dense_mask_bruteforce(lengths, is_global):
    rng = np.random.default_rng(sum(lengths) + is_global)
    T, nh, d, window = sum(lengths), 2, 16, 64
    q, k, v = (rng.standard_normal((T, nh, d)) for _ in range(3))
    want = _dense_attention(q, k, v, _dense_mask(lengths, window, is_global))
    got = np.zeros_like(q)
    start = 0
    for n in lengths:
        sl = slice(start, start + n)
        got[sl] = oracle.attention_text(q[sl], k[sl], v[sl], is_global, window, q_chunk=37)
        start += n
    np.testing.assert_allclose(got, want, atol=1e-12)


def test_attention_uniform_scores_average_the_window():
    # q = 0 makes every allowed score equal, so the output is the plain mean
    # of the allowed values: keys max(0, i-w) .. min(L-1, i+w).
    L, w = 200, 64
    rng = np.random.default_rng(4)
    v = rng.standard_normal((L, 1, 8))
    z = np.zeros((L, 1, 8))
    out = oracle.attention_text(z, z, v, False, w)
    for i in (0, 1, 63, 64, 65, 100, 135, 136, 199):
        lo, hi = max(0, i - w), min(L - 1, i + w)
        np.testing.assert_allclose(out[i, 0], v[lo:hi + 1, 0].mean(axis=0), atol=1e-12)
    out_g = oracle.attention_text(z, z, v, True, w)
    np.testing.assert_allclose(out_g[17, 0], v[:, 0].mean(axis=0), atol=1e-12)


# --------------------------------------------------------------------------
# Pooling
# --------------------------------------------------------------------------

def test_pool_l2_unit_norm_and_mean_direction():
    rng = np.random.default_rng(6)
    s = rng.standard_normal((13, 32))
    p = oracle.pool_l2(s)
    assert abs(np.linalg.norm(p) - 1.0) < 1e-14
    m = s.sum(axis=0)                         # same direction as the mean
    np.testing.assert_allclose(p, m / np.linalg.norm(m), atol=1e-14)
    np.testing.assert_array_equal(oracle.pool_l2(np.zeros((3, 4))), np.zeros(4))


# --------------------------------------------------------------------------
# The whole encoder
# --------------------------------------------------------------------------

MICRO = synth.Shape(n_layers=4, hidden=8, n_heads=2, head_dim=4, intermediate=6, vocab=16,
                    global_every=3, window=2, rope_base_global=50.0, rope_base_local=7.0, ln_eps=1e-5)


def _brute_encode(ids, lengths, w, shape, tokens=False):
    """Scalar loops over the packed sequence: every step written out from the
    definition, with a dense same-text/window mask and complex RoPE.  With
    ``tokens`` it returns the per-token unit vectors (projected when the shape
    has a projection) instead of the pooled ones."""
    H, nh, d, I = shape.hidden, shape.n_heads, shape.head_dim, shape.intermediate
    T = len(ids)
    text, pos = [], []
    for j, n in enumerate(lengths):
        text += [j] * n
        pos += list(range(n))

    def ln(row, g):
        m = sum(row) / H
        var = sum((r - m) ** 2 for r in row) / H
        return [(row[c] - m) / math.sqrt(var + shape.ln_eps) * float(g[c]) for c in range(H)]

    def matvec(W, row):
        return [sum(float(W[r][c]) * row[c] for c in range(len(row))) for r in range(len(W))]

    def phi(a):
        return 0.5 * math.erfc(-a / math.sqrt(2.0))

    x = [[float(w.tok_emb[i][c]) for c in range(H)] for i in ids]
    if shape.emb_norm:
        x = [ln(row, w.ln_emb) for row in x]
    for l in range(shape.n_layers):
        glob = l % shape.global_every == 0
        base = shape.rope_base_global if glob else shape.rope_base_local
        qkv = [matvec(w.wqkv[l], ln(x[t], w.ln_attn[l])) for t in range(T)]
        q = [[0.0] * H for _ in range(T)]
        k = [[0.0] * H for _ in range(T)]
        for t in range(T):
            for h in range(nh):
                for j in range(d // 2):
                    rot = cmath.exp(1j * pos[t] * base ** (-2.0 * j / d))
                    for dst, off in ((q, 0), (k, H)):
                        z = complex(qkv[t][off + h * d + j], qkv[t][off + h * d + j + d // 2]) * rot
                        dst[t][h * d + j] = z.real
                        dst[t][h * d + j + d // 2] = z.imag
        o = [[0.0] * H for _ in range(T)]
        for t in range(T):
            for h in range(nh):
                keys = [s for s in range(T) if text[s] == text[t]
                        and (glob or abs(pos[s] - pos[t]) <= shape.window)]
                sc = [sum(q[t][h * d + c] * k[s][h * d + c] for c in range(d)) / math.sqrt(d) for s in keys]
                mx = max(sc)
                e = [math.exp(a - mx) for a in sc]
                tot = sum(e)
                for c in range(d):
                    o[t][h * d + c] = sum(e[i] / tot * qkv[s][2 * H + h * d + c] for i, s in enumerate(keys))
        for t in range(T):
            y = matvec(w.wo[l], o[t])
            x[t] = [x[t][c] + y[c] for c in range(H)]
        for t in range(T):
            u = matvec(w.wi[l], ln(x[t], w.ln_mlp[l]))
            z = [u[c] * phi(u[c]) * u[I + c] for c in range(I)]
            y = matvec(w.wo_ffn[l], z)
            x[t] = [x[t][c] + y[c] for c in range(H)]
    if shape.final_norm:
        x = [ln(row, w.ln_final) for row in x]
    if tokens:
        rows = [matvec(w.w_proj, row) if shape.proj_dim else row for row in x]
        return np.array([[a / math.sqrt(sum(b * b for b in row)) for a in row] for row in rows])
    out = []
    start = 0
    for n in lengths:
        m = [sum(x[t][c] for t in range(start, start + n)) / n for c in range(H)]
        nrm = math.sqrt(sum(a * a for a in m))
        out.append([a / nrm for a in m])
        start += n
    return np.array(out)


def _micro_weights(seed=0, std=0.5):
    # a larger std than the real recipe so that attention is far from uniform
    return synth.make_weights(MICRO, seed=seed, std=std)


@pytest.mark.parametrize("variant", ["fp32", "bf16"])
def test_encoder_matches_scalar_bruteforce(variant):
    lengths = [1, 3, 7, 5]
    w = _micro_weights()
    ids, cu = synth.make_batch(lengths, MICRO.vocab, seed=3)
    model = oracle.OracleModel(w, MICRO, variant)
    got = oracle.encode_packed(ids, cu, model)
    if variant == "bf16":
        for name in ("wqkv", "wo", "wi", "wo_ffn", "ln_attn", "ln_mlp"):
            setattr(w, name, [oracle.round_to_bf16(a) for a in getattr(w, name)])
        w.tok_emb = oracle.round_to_bf16(w.tok_emb)
    want = _brute_encode(ids, lengths, w, MICRO)
    np.testing.assert_allclose(got, want, atol=1e-12)


MICRO_EXT = synth.Shape(**{**MICRO.as_dict(), "emb_norm": True, "final_norm": True, "proj_dim": 5})


def _rounded(w, variant):
    """The weights as the bf16 variant stores them (for the brute force)."""
    if variant == "bf16":
        for name in ("wqkv", "wo", "wi", "wo_ffn", "ln_attn", "ln_mlp"):
            setattr(w, name, [oracle.round_to_bf16(a) for a in getattr(w, name)])
        for name in ("tok_emb", "ln_emb", "ln_final", "w_proj"):
            if getattr(w, name) is not None:
                setattr(w, name, oracle.round_to_bf16(getattr(w, name)))
    return w


@pytest.mark.parametrize("variant", ["fp32", "bf16"])
def test_optional_norms_and_token_output_match_scalar_bruteforce(variant):
    # embedding norm, final norm, and the per-token projected unit vectors
    lengths = [1, 3, 7, 5]
    w = synth.make_weights(MICRO_EXT, seed=7, std=0.5)
    ids, cu = synth.make_batch(lengths, MICRO.vocab, seed=8)
    model = oracle.OracleModel(w, MICRO_EXT, variant)
    pooled = oracle.encode_packed(ids, cu, model)
    toks = oracle.encode_packed_tokens(ids, cu, model)
    assert toks.shape == (sum(lengths), MICRO_EXT.proj_dim)
    w = _rounded(w, variant)
    np.testing.assert_allclose(pooled, _brute_encode(ids, lengths, w, MICRO_EXT), atol=1e-12)
    np.testing.assert_allclose(toks, _brute_encode(ids, lengths, w, MICRO_EXT, tokens=True), atol=1e-12)


def test_optional_norms_change_the_result_and_draws_stay_put():
    # the optional parts are drawn after the layers: the shared weights are identical
    base = synth.make_weights(MICRO, seed=7, std=0.5)
    ext = synth.make_weights(MICRO_EXT, seed=7, std=0.5)
    np.testing.assert_array_equal(base.tok_emb, ext.tok_emb)
    for l in range(MICRO.n_layers):
        np.testing.assert_array_equal(base.wo_ffn[l], ext.wo_ffn[l])
    ids, cu = synth.make_batch([6, 4], MICRO.vocab, seed=9)
    a = oracle.encode_packed(ids, cu, oracle.OracleModel(base, MICRO))
    b = oracle.encode_packed(ids, cu, oracle.OracleModel(ext, MICRO_EXT))
    assert np.abs(a - b).max() > 1e-3


def test_token_output_closed_forms():
    # no projection: a one-token text's token vector is its pooled vector;
    # identity projection = no projection; every token vector has unit norm
    shape = synth.TINY
    w = synth.make_weights(shape, seed=10)
    ids, cu = synth.make_batch([1, 9, 30], shape.vocab, seed=11)
    model = oracle.OracleModel(w, shape)
    toks = oracle.encode_packed_tokens(ids, cu, model)
    np.testing.assert_allclose(np.linalg.norm(toks, axis=1), 1.0, atol=1e-14)
    np.testing.assert_allclose(toks[0], oracle.encode_packed(ids, cu, model)[0], atol=1e-14)
    eye = synth.Shape(**{**shape.as_dict(), "proj_dim": shape.hidden})
    w.w_proj = np.eye(shape.hidden, dtype=np.float32)
    np.testing.assert_allclose(oracle.encode_packed_tokens(ids, cu, oracle.OracleModel(w, eye)), toks, atol=1e-14)


def test_encoder_zero_projections_is_mean_embedding():
    w = synth.make_weights(synth.TINY, seed=1)
    for l in range(synth.TINY.n_layers):
        w.wo[l][:] = 0
        w.wo_ffn[l][:] = 0
    ids, cu = synth.make_batch([5, 9], synth.TINY.vocab, seed=2)
    got = oracle.encode_packed(ids, cu, oracle.OracleModel(w, synth.TINY))
    for j in range(2):
        m = w.tok_emb[ids[cu[j]:cu[j + 1]]].astype(np.float64).mean(axis=0)
        np.testing.assert_allclose(got[j], m / np.linalg.norm(m), atol=1e-12)


def test_encoder_single_token_text_closed_form():
    # One token: RoPE at position 0 is the identity and softmax over one key
    # is 1, so each layer is x += Wo (Wv LN(x)), x += Wo_ffn GeGLU(Wi LN(x)).
    shape = synth.TINY
    w = synth.make_weights(shape, seed=4)
    H, I = shape.hidden, shape.intermediate
    tok = 77
    x = w.tok_emb[tok].astype(np.float64)
    for l in range(shape.n_layers):
        n = oracle.layernorm(x[None], w.ln_attn[l], shape.ln_eps)[0]
        vv = w.wqkv[l][2 * H:].astype(np.float64) @ n
        x = x + w.wo[l].astype(np.float64) @ vv
        n = oracle.layernorm(x[None], w.ln_mlp[l], shape.ln_eps)[0]
        u = w.wi[l].astype(np.float64) @ n
        x = x + w.wo_ffn[l].astype(np.float64) @ (u[:I] * np.array([_phi(a) for a in u[:I]]) * u[I:])
    got = oracle.encode_text(np.array([tok]), oracle.OracleModel(w, shape))
    np.testing.assert_allclose(got, x / np.linalg.norm(x), atol=1e-12)


def _phi(a):
    return 0.5 * math.erfc(-a / math.sqrt(2.0))


def test_window_layers_equal_global_on_short_texts():
    # With |i - j| <= 64 for every pair (L <= 65) and equal RoPE bases, a
    # window layer computes exactly what a global layer does.
    base = synth.TINY
    every = synth.Shape(**{**base.as_dict(), "global_every": 1, "rope_base_local": base.rope_base_global})
    mixed = synth.Shape(**{**base.as_dict(), "rope_base_local": base.rope_base_global})
    w = synth.make_weights(base, seed=5)
    ids, cu = synth.make_batch([65, 12], base.vocab, seed=6)
    a = oracle.encode_packed(ids, cu, oracle.OracleModel(w, every))
    b = oracle.encode_packed(ids, cu, oracle.OracleModel(w, mixed))
    np.testing.assert_allclose(a, b, atol=1e-13)
    # ... and a 66-token text does see the difference
    ids2, cu2 = synth.make_batch([66], base.vocab, seed=6)
    a2 = oracle.encode_packed(ids2, cu2, oracle.OracleModel(w, every))
    b2 = oracle.encode_packed(ids2, cu2, oracle.OracleModel(w, mixed))
    assert np.abs(a2 - b2).max() > 1e-9


def test_encoder_outputs_unit_norm_and_self_similarity():
    w = synth.make_weights(synth.TINY, seed=0)
    ids, cu = synth.make_batch(synth.TINY_LENGTHS, synth.TINY.vocab, seed=0)
    e = oracle.encode_packed(ids, cu, oracle.OracleModel(w, synth.TINY))
    np.testing.assert_allclose(np.linalg.norm(e, axis=1), 1.0, atol=1e-14)
    sim = e @ e.T
    np.testing.assert_allclose(np.diag(sim), 1.0, atol=1e-14)
    np.testing.assert_allclose(sim, sim.T, atol=0)
    assert np.all(np.abs(sim) <= 1.0 + 1e-14)
    # same structure as the similarity matrix the page prints
    page = np.loadtxt(os.path.join(GOLDEN, "ruri_sim_matrix.txt"))
    np.testing.assert_allclose(np.diag(page), 1.0)
    np.testing.assert_allclose(page, page.T)
