"""Each step of the pass, run through the C ABI on the GPU, against the oracle.

Shapes: the tiny encoder (hidden 256), an odd one (hidden 384, 6 heads,
GeGLU width 640) whose projections exercise the 128-column GEMM tiles, and a
wide one (GeGLU width 1280) whose long-K output projection runs on 192-column
tiles, and a narrow one (hidden 768, GeGLU width 1024) whose Wqkv is the
largest weight staged on load; token
counts are ragged (not multiples of the 128-row tiles) and texts straddle
tile edges.
"""
import numpy as np
import pytest

import oracle
from text_embedding_encoder_gb300 import binding, synth

torch = pytest.importorskip("torch")
from gpu_util import act_dtype, assert_step_close, dev, make_encoder, to_np  # noqa: E402

pytestmark = pytest.mark.gpu

ODD = synth.Shape(n_layers=2, hidden=384, n_heads=6, head_dim=64, intermediate=640, vocab=1000)
# a long GeGLU width: the feed-forward output projection (K = 1280) runs on 192-column tiles
WIDE = synth.Shape(n_layers=2, hidden=384, n_heads=6, head_dim=64, intermediate=1280, vocab=1000)
# a GeGLU narrower than 1.5 x hidden: Wqkv is the largest weight staged on load
NARROW = synth.Shape(n_layers=2, hidden=768, n_heads=12, head_dim=64, intermediate=1024, vocab=1000)
LENGTHS = [1, 2, 63, 64, 65, 66, 129, 127, 3, 300]   # 820 tokens


@pytest.fixture(scope="module", params=[("tiny", "fp32"), ("tiny", "bf16"), ("odd", "bf16"), ("odd", "fp32"),
                                        ("wide", "bf16"), ("narrow", "bf16")],
                ids=lambda p: f"{p[0]}-{p[1]}")
def setup(request, lib):
    name, dt = request.param
    shape = {"tiny": synth.TINY, "odd": ODD, "wide": WIDE, "narrow": NARROW}[name]
    w = synth.make_weights(shape, seed=11, std=0.05)
    enc = make_encoder(shape, dt, w, max_tokens=1024, max_texts=64)
    model = oracle.OracleModel(w, shape, dt)
    ids, cu = synth.make_batch(LENGTHS, shape.vocab, seed=12)
    yield shape, dt, w, enc, model, ids, cu
    enc.close()


def _positions(cu):
    return np.concatenate([np.arange(b - a) for a, b in zip(cu[:-1], cu[1:])])


def _act(x, dt):
    """Activation input as the GPU sees it, and as the oracle sees it (same values)."""
    t = dev(x.astype(np.float32), act_dtype(dt))
    return t, to_np(t)


def test_embed_and_positions(setup):
    shape, dt, w, enc, model, ids, cu = setup
    T = len(ids)
    x = torch.empty(T, shape.hidden, device="cuda")
    enc.op("tee_op_embed", dev(ids), T, x, 0)
    pos = torch.empty(T, dtype=torch.int32, device="cuda")
    enc.op("tee_op_positions", dev(cu), cu, len(cu) - 1, pos, 0)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(to_np(x), model.tok_emb[ids].astype(np.float64))
    np.testing.assert_array_equal(pos.cpu().numpy(), _positions(cu))
    assert enc.device_status() == 0


@pytest.mark.parametrize("which", [0, 1])
def test_layernorm(setup, which):
    shape, dt, w, enc, model, ids, cu = setup
    T = len(ids)
    rng = np.random.default_rng(1)
    x = (rng.standard_normal((T, shape.hidden)) * 0.7 + 0.3).astype(np.float32)
    y = torch.empty(T, shape.hidden, dtype=act_dtype(dt), device="cuda")
    layer = shape.n_layers - 1
    enc.op("tee_op_layernorm", layer, which, dev(x), y, T, 0)
    gamma = (model.ln_attn if which == 0 else model.ln_mlp)[layer]
    assert_step_close(to_np(y), oracle.layernorm(x, gamma, shape.ln_eps), dt)


@pytest.mark.parametrize("layer", [0, 1])
def test_qkv_with_rope(setup, layer):
    shape, dt, w, enc, model, ids, cu = setup
    T, H = len(ids), shape.hidden
    rng = np.random.default_rng(2)
    y_t, y = _act(rng.standard_normal((T, H)), dt)
    pos = dev(_positions(cu).astype(np.int32))
    out = torch.empty(T, 3 * H, dtype=act_dtype(dt), device="cuda")
    enc.op("tee_op_qkv", layer, y_t, pos, out, T, 0)
    qkv = model.linear("wqkv", layer, y)
    base = shape.rope_base_global if oracle.layer_is_global(layer, shape) else shape.rope_base_local
    p = _positions(cu)
    nh = shape.n_heads
    q = oracle.apply_rope(qkv[:, :H].reshape(T, nh, 64), p, base).reshape(T, H)
    k = oracle.apply_rope(qkv[:, H:2 * H].reshape(T, nh, 64), p, base).reshape(T, H)
    ref = np.concatenate([q, k, qkv[:, 2 * H:]], axis=1)
    assert_step_close(to_np(out), ref, dt)


@pytest.mark.parametrize("layer", [0, 1])
def test_attention(setup, layer):
    shape, dt, w, enc, model, ids, cu = setup
    T, H, nh = len(ids), shape.hidden, shape.n_heads
    rng = np.random.default_rng(3 + layer)
    qkv_t, qkv = _act(rng.standard_normal((T, 3 * H)) * 1.5, dt)
    o = torch.empty(T, H, dtype=act_dtype(dt), device="cuda")
    enc.op("tee_op_attention", layer, qkv_t, dev(cu), cu, len(cu) - 1, o, 0)
    is_g = oracle.layer_is_global(layer, shape)
    ref = np.zeros((T, H))
    for a, b in zip(cu[:-1], cu[1:]):
        sl = slice(a, b)
        q = qkv[sl, :H].reshape(-1, nh, 64)
        k = qkv[sl, H:2 * H].reshape(-1, nh, 64)
        v = qkv[sl, 2 * H:].reshape(-1, nh, 64)
        ref[sl] = oracle.attention_text(q, k, v, is_g, shape.window).reshape(-1, H)
    assert_step_close(to_np(o), ref, dt)


def test_out_proj_and_ffn(setup):
    shape, dt, w, enc, model, ids, cu = setup
    T, H, I = len(ids), shape.hidden, shape.intermediate
    rng = np.random.default_rng(5)
    layer = 1
    x0 = rng.standard_normal((T, H)).astype(np.float32)
    o_t, o = _act(rng.standard_normal((T, H)), dt)
    x = dev(x0)
    enc.op("tee_op_out_proj", layer, o_t, x, T, 0)
    ref = x0.astype(np.float64) + model.linear("wo", layer, o)
    assert_step_close(to_np(x), ref, "fp32", fp32_atol=2e-5 if dt == "fp32" else 3e-3)

    y_t, y = _act(rng.standard_normal((T, H)), dt)
    z = torch.empty(T, I, dtype=act_dtype(dt), device="cuda")
    enc.op("tee_op_ffn_in", layer, y_t, z, T, 0)
    assert_step_close(to_np(z), oracle.geglu(model.linear("wi", layer, y), I), dt)

    z_t, zz = _act(rng.standard_normal((T, I)), dt)
    x = dev(x0)
    enc.op("tee_op_ffn_out", layer, z_t, x, T, 0)
    ref = x0.astype(np.float64) + model.linear("wo_ffn", layer, zz)
    assert_step_close(to_np(x), ref, "fp32", fp32_atol=2e-5 if dt == "fp32" else 3e-3)


def test_pool_l2(setup):
    shape, dt, w, enc, model, ids, cu = setup
    T, H = len(ids), shape.hidden
    rng = np.random.default_rng(6)
    x = rng.standard_normal((T, H)).astype(np.float32)
    out = torch.empty(len(cu) - 1, H, device="cuda")
    enc.op("tee_op_pool_l2", dev(x), dev(cu), cu, len(cu) - 1, out, 0)
    ref = np.stack([oracle.pool_l2(x[a:b]) for a, b in zip(cu[:-1], cu[1:])])
    np.testing.assert_allclose(to_np(out), ref, atol=2e-6)


# ---------------------------------------------------------------------------
# integer path
# ---------------------------------------------------------------------------

@pytest.fixture(scope="module")
def w8a8(lib):
    shape = ODD
    w = synth.make_weights(shape, seed=21, outliers=True)
    enc = make_encoder(shape, "w8a8", w, max_tokens=1024, max_texts=64)
    yield shape, w, enc
    enc.close()


def test_quant_rows7_bit_exact(w8a8):
    shape, w, enc = w8a8
    rng = np.random.default_rng(7)
    M, K = 517, shape.intermediate
    x = (rng.standard_normal((M, K)) * rng.uniform(0.01, 30, (M, 1))).astype(np.float32)
    x[:, 17] *= 20.0
    x[3] = 0.0
    x[5, :4] = [63.0, 0.5, 1.5, 2.5]
    x[5, 4:] = 0.0
    q = torch.empty(M, K, dtype=torch.int8, device="cuda")
    s = torch.empty(M, device="cuda")
    enc.op("tee_op_quant_rows7", dev(x), M, K, q, s, 0)
    q_ref, s_ref = oracle.quantize_rows7(x)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(q.cpu().numpy(), q_ref)
    np.testing.assert_array_equal(s.cpu().numpy().view(np.uint32), s_ref.view(np.uint32))


@pytest.mark.parametrize("which,name", [(0, "wqkv"), (1, "wo"), (2, "wi"), (3, "wo_ffn")])
def test_weight_codes_and_block_sums_bit_exact(w8a8, which, name):
    shape, w, enc = w8a8
    layer = 1
    Wf = getattr(w, name)[layer]
    N, K = Wf.shape
    q_ref, d_ref = oracle.quantize_weight_blocks(Wf)
    q_gpu = np.empty((N, K), np.int8)
    d_gpu = np.empty((N, K // 32), np.float32)
    enc.check(enc.lib.tee_weight_codes(enc.ctx, layer, which, q_gpu.ctypes.data, d_gpu.ctypes.data))
    np.testing.assert_array_equal(q_gpu, q_ref)
    np.testing.assert_array_equal(d_gpu.view(np.uint32), d_ref.view(np.uint32))

    rng = np.random.default_rng(8 + which)
    M = 141
    qa, _ = oracle.quantize_rows7((rng.standard_normal((M, K)) * 3).astype(np.float32))
    qa[0, :] = 63
    parts = torch.empty(M, N, K // 32, dtype=torch.int32, device="cuda")
    enc.op("tee_op_w8a8_partials", layer, which, dev(qa), M, parts, 0)
    ref = oracle.int_block_partials(qa, q_ref)
    np.testing.assert_array_equal(parts.cpu().numpy().astype(np.int64), ref)


# ---------------------------------------------------------------------------
# the projection GEMM on arbitrary shapes (tile tails, both epilogues, every
# tile width and the 2-CTA weight multicast)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("M,N,K", [(1, 128, 64), (259, 384, 192), (1000, 256, 768), (513, 768, 3072),
                                   (700, 2304, 768)])
@pytest.mark.parametrize("epi", [0, 1])
def test_gemm_bf16_shapes(lib, M, N, K, epi):
    enc = binding.Encoder(synth.TINY, "bf16", max_tokens=16, max_texts=4)
    rng = np.random.default_rng(M + N + K)
    a = dev(rng.standard_normal((M, K)).astype(np.float32), torch.bfloat16)
    w = dev((rng.standard_normal((N, K)) * 0.05).astype(np.float32), torch.bfloat16)
    ref = to_np(a) @ to_np(w).T
    if epi == 0:
        c = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
        enc.op("tee_op_gemm_bf16", a, w, c, M, N, K, 0, 0)
        assert_step_close(to_np(c), ref, "bf16")
    else:
        c0 = rng.standard_normal((M, N)).astype(np.float32)
        c = dev(c0)
        enc.op("tee_op_gemm_bf16", a, w, c, M, N, K, 1, 0)
        np.testing.assert_allclose(to_np(c), c0.astype(np.float64) + ref, atol=2e-3 * max(1.0, np.abs(ref).max()))
    enc.close()


# a context of the 310m widths (one layer)
W768 = synth.Shape(n_layers=1, hidden=768, n_heads=12, head_dim=64, intermediate=3072, vocab=16)


def _residual_gemm_twice(M, N, K, seed):
    """C += A W^T through tee_op_gemm_bf16 in a W768 context, twice from the
    same C: the two results must be bit-identical (every output element is
    summed in one fixed order).  Returns (result, A, W, C0) as torch tensors."""
    enc = binding.Encoder(W768, "bf16", max_tokens=M, max_texts=4)
    g = torch.Generator(device="cuda").manual_seed(seed)
    a = torch.randn(M, K, device="cuda", generator=g).to(torch.bfloat16)
    w = (torch.randn(N, K, device="cuda", generator=g) * 0.05).to(torch.bfloat16)
    c0 = torch.randn(M, N, device="cuda", generator=g)
    outs = []
    for _ in range(2):
        c = c0.clone()
        enc.op("tee_op_gemm_bf16", a, w, c, M, N, K, 1, 0)
        torch.cuda.synchronize()
        outs.append(c)
    enc.close()
    assert torch.equal(outs[0], outs[1])
    return outs[0], a, w, c0


def _check_residual(c, a, w, c0):
    ref = c0.double() + a.double() @ w.double().T
    err = (c.double() - ref).abs().max().item()
    assert err <= 2e-3 * max(1.0, (ref - c0.double()).abs().max().item()), err


@pytest.mark.parametrize("M", [2048, 24000, 32768])
def test_gemm_residual_short_k_tile_choices(lib, M):
    # the attention out-projection shape at row counts whose wave model picks
    # 128-column tiles (2048) and 192-column tiles (24000, 32768), one CTA each
    _check_residual(*_residual_gemm_twice(M, 768, 768, M + 1))


@pytest.mark.parametrize("M", [2048, 8192, 20000, 32768])
def test_gemm_residual_long_k_tile_choices(lib, M):
    # the FFN out-projection shape at row counts whose wave model picks single
    # CTAs on 128 columns (2048), CTA pairs on 192 (8192) and on 256 (20000,
    # 32768: 384 pair tiles, the pass's own launch)
    _check_residual(*_residual_gemm_twice(M, 768, 3072, M))


def test_step_entry_points_reject_unaligned_and_null_buffers(lib):
    # every check returns before anything is launched; the context stays usable
    shape = synth.TINY
    enc = make_encoder(shape, "bf16", synth.make_weights(shape, seed=0), max_tokens=64, max_texts=4)
    T, H = 16, shape.hidden
    cu = np.array([0, T], np.int32)
    buf = torch.zeros(3 * T * shape.intermediate + 64, dtype=torch.float32, device="cuda")
    good = buf.data_ptr()
    bad = good + 4                      # 4-byte aligned, not 16
    d_cu, ids, pos = dev(cu), dev(np.ones(T, np.int32)), dev(np.zeros(T, np.int32))
    calls = [
        ("tee_op_embed", lambda p: (ids, T, p, 0)),
        ("tee_op_layernorm", lambda p: (0, 0, p, good, T, 0)),
        ("tee_op_layernorm", lambda p: (0, 0, good, p, T, 0)),
        ("tee_op_qkv", lambda p: (0, p, pos, good, T, 0)),
        ("tee_op_attention", lambda p: (0, p, d_cu, cu, 1, good, 0)),
        ("tee_op_out_proj", lambda p: (0, p, good, T, 0)),
        ("tee_op_ffn_in", lambda p: (0, good, p, T, 0)),
        ("tee_op_ffn_out", lambda p: (0, good, p, T, 0)),
        ("tee_op_pool_l2", lambda p: (p, d_cu, cu, 1, good, 0)),
    ]
    for name, args in calls:
        for p in (bad, 0):
            with pytest.raises(binding.TeeError) as e:
                enc.op(name, *args(p))
            assert e.value.code == binding.TEE_EINVAL, (name, p)
    with pytest.raises(binding.TeeError) as e:   # int32 arrays: 4-byte alignment
        enc.op("tee_op_positions", d_cu, cu, 1, good + 2, 0)
    assert e.value.code == binding.TEE_EINVAL
    x = torch.empty(T, H, device="cuda")
    enc.op("tee_op_embed", ids, T, x, 0)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(to_np(x), np.broadcast_to(to_np(x)[:1], (T, H)))   # every id is 1
    enc.close()


def test_geglu_epilogue_gelu_dense_range(lib):
    """The GeGLU epilogue of the tensor-core feed-forward projection evaluates
    GELU with its own erf (Abramowitz & Stegun 7.1.26 on the hardware
    reciprocal and exp2).  Checked over a dense range against the oracle's
    GELU (scipy erf in fp64): the formula's own error (|erf error| <= 1.5e-7,
    times |a| / 2 in GELU) plus the half-ulp rounding of the fp32 result."""
    rng = np.random.default_rng(5)
    a = np.concatenate([np.linspace(-10.0, 10.0, 1_000_001), rng.uniform(-10.0, 10.0, 1_000_000),
                        np.array([0.0, -0.0, 1e-30, -1e-30, 1e-8, -1e-8, 12.0, -12.0, 14.0, -14.0, 30.0, -30.0])])
    a = a.astype(np.float32)
    d_a = dev(a)
    d_y = torch.full_like(d_a, float("nan"))
    rc = lib.tee_selftest_gelu(d_a.data_ptr(), d_y.data_ptr(), a.size, 0)
    assert rc == binding.TEE_OK, lib.tee_last_error(None).decode()
    torch.cuda.synchronize()
    got = to_np(d_y)
    ref = oracle.gelu(a.astype(np.float64))
    err = np.abs(got - ref)
    bound = 6e-7 + 2.0 ** -24 * np.abs(ref)
    worst = int(np.argmax(err - bound))
    print(f"GELU epilogue: max abs err {err.max():.3e} (at a = {a[int(np.argmax(err))]:.4f})")
    assert np.all(err <= bound), (float(a[worst]), float(err[worst]), float(bound[worst]))
    assert np.all(got[a == 0.0] == 0.0)
    # misaligned buffers are refused before any launch
    assert lib.tee_selftest_gelu(d_a.data_ptr() + 2, d_y.data_ptr(), 4, 0) == binding.TEE_EINVAL
