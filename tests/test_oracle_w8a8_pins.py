"""Pins for the oracle's integer (W8A8) path.

Hand-worked quantiser cases (ties to even, clamping, zero rows), the integer
block sums against pure-Python integer loops, and the dequantised product
against the float product within the bound that the two rounding errors
allow.
"""
import numpy as np

import oracle
from oracle import w8a8


def test_quantize_rows7_hand_cases():
    x = np.array([
        [63.0, 0.5, 1.5, 2.5, -0.5, -62.5, 31.5, 0.0],   # s = 1: ties go to even
        [0.0] * 8,                                       # zero row
        [-2.0, 1.0, 0.0, 0.0, 0.0, 0.0, 0.0, 0.0],         # s = 2/63
    ], dtype=np.float32)
    q, s = oracle.quantize_rows7(x)
    assert s[0] == np.float32(1.0)
    assert q[0].tolist() == [63, 0, 2, 2, 0, -62, 32, 0]
    assert s[1] == 0.0 and not q[1].any()
    assert s[2] == np.float32(2.0) / np.float32(63.0)
    assert q[2, 0] == -63
    # fp32 decides: s rounds up slightly, so 1 / s = 31.499998 and the code is
    # 31, not the 32 that exact arithmetic (31.5, tie to even) would give.
    assert np.float32(1.0) / s[2] == np.float32(31.499998)
    assert q[2, 1] == 31


def test_quantize_rows7_range_and_error():
    rng = np.random.default_rng(0)
    x = (rng.standard_normal((64, 96)) * rng.uniform(0.01, 10, (64, 1))).astype(np.float32)
    q, s = oracle.quantize_rows7(x)
    assert np.abs(q.astype(int)).max() <= 63
    assert np.all(np.abs(q).max(axis=1) == 63)            # the row maximum maps to +-63
    err = np.abs(q.astype(np.float64) * s[:, None] - x)
    assert np.all(err <= s[:, None] * (0.5 + 1e-6))


def test_quantize_weight_blocks_hand_cases():
    w = np.zeros((2, 64), np.float32)
    w[0, :32] = np.linspace(-127, 127, 32)
    w[0, 32] = 0.5
    w[0, 33] = 1.5
    w[0, 34] = 127.0
    w[1, 40] = -3.0
    q, d = oracle.quantize_weight_blocks(w)
    assert d.shape == (2, 2)
    assert d[0, 0] == 1.0 and d[0, 1] == 1.0
    np.testing.assert_array_equal(q[0, :32], np.rint(np.linspace(-127, 127, 32)).astype(np.int8))
    assert q[0, 32] == 0 and q[0, 33] == 2 and q[0, 34] == 127
    assert d[1, 0] == 0.0 and not q[1, :32].any()
    assert q[1, 40] == -127 and d[1, 1] == np.float32(3.0) / np.float32(127.0)


def test_quantize_weight_blocks4_hand_cases():
    # 4-bit blocks: d = max|w| / 7, codes rint(w / d) clamped to +-7, ties to even
    w = np.zeros((2, 64), np.float32)
    w[0, :32] = np.linspace(-7, 7, 32)
    w[0, 32] = 0.5        # 0.5 / 1 -> 0 (tie to even)
    w[0, 33] = 2.5        # -> 2
    w[0, 34] = 3.5        # -> 4
    w[0, 35] = 7.0        # the block maximum: d = 1
    w[1, 40] = -3.0       # alone in its block: d = 3/7, code -7
    q, d = oracle.quantize_weight_blocks4(w)
    assert d[0, 0] == 1.0 and d[0, 1] == 1.0
    np.testing.assert_array_equal(q[0, :32], np.rint(np.linspace(-7, 7, 32)).astype(np.int8))
    assert q[0, 32] == 0 and q[0, 33] == 2 and q[0, 34] == 4 and q[0, 35] == 7
    assert d[1, 0] == 0.0 and not q[1, :32].any()
    assert q[1, 40] == -7 and d[1, 1] == np.float32(3.0) / np.float32(7.0)


def test_quantize_weight_blocks4_range_and_error():
    rng = np.random.default_rng(5)
    w = (rng.standard_normal((16, 128)) * rng.uniform(0.01, 3, (16, 1))).astype(np.float32)
    q, d = oracle.quantize_weight_blocks4(w)
    assert q.min() >= -7 and q.max() <= 7
    # every block reaches +-7 at its maximum, and the rounding error is at most d / 2
    blocks = np.abs(q.reshape(16, 4, 32)).max(axis=2)
    np.testing.assert_array_equal(blocks, 7)
    err = np.abs(w.reshape(16, 4, 32) - q.reshape(16, 4, 32) * d[:, :, None])
    assert np.all(err <= d[:, :, None] / 2 * (1 + 1e-6))


def test_quantize_weight_blocks6_hand_cases():
    # 6-bit blocks: d = max|w| / 31, codes rint(w / d) clamped to +-31, ties to even
    w = np.zeros((2, 64), np.float32)
    w[0, :32] = np.linspace(-31, 31, 32)   # d = 1: codes are the rounded values themselves
    w[0, 32] = 0.5        # tie -> 0 (even)
    w[0, 33] = 1.5        # tie -> 2 (even)
    w[0, 34] = 14.5       # tie -> 14 (even)
    w[0, 35] = 31.0       # the block maximum: d = 1
    w[0, 36] = -30.5      # tie -> -30 (even)
    w[1, 40] = -3.0       # alone in its block: d = 3/31, code -31
    q, d = oracle.quantize_weight_blocks6(w)
    assert d[0, 0] == 1.0 and d[0, 1] == 1.0 and d[1, 0] == 0.0
    np.testing.assert_array_equal(q[0, :32], np.rint(np.linspace(-31, 31, 32)).astype(np.int8))
    assert q[0, 32] == 0 and q[0, 33] == 2 and q[0, 34] == 14 and q[0, 35] == 31 and q[0, 36] == -30
    np.testing.assert_array_equal(q[1, :32], 0)                            # an all-zero block
    assert q[1, 40] == -31 and d[1, 1] == np.float32(3.0) / np.float32(31.0)


def test_quantize_weight_blocks6_range_and_error():
    rng = np.random.default_rng(6)
    w = (rng.standard_normal((16, 128)) * rng.uniform(0.001, 1.0, (16, 1))).astype(np.float32)
    q, d = oracle.quantize_weight_blocks6(w)
    assert q.min() >= -31 and q.max() <= 31
    # every block reaches +-31 at its maximum, and the rounding error is at most d / 2
    np.testing.assert_array_equal(np.abs(q.reshape(16, 4, 32)).max(axis=2), 31)
    err = np.abs(w.reshape(16, 4, 32) - q.reshape(16, 4, 32) * d[:, :, None])
    assert np.all(err <= d[:, :, None] / 2 * (1 + 1e-6))
    # finer than 4-bit blocks, coarser than 8-bit ones on the same weights
    e4 = np.abs(w - oracle.quantize_weight_blocks4(w)[0] * np.repeat(oracle.quantize_weight_blocks4(w)[1], 32, 1))
    e8 = np.abs(w - oracle.quantize_weight_blocks(w)[0] * np.repeat(oracle.quantize_weight_blocks(w)[1], 32, 1))
    e6 = np.abs(w - q * np.repeat(d, 32, 1))
    assert e8.mean() < e6.mean() < e4.mean()


def test_int_block_partials_against_integer_loops():
    rng = np.random.default_rng(1)
    M, N, K = 5, 4, 96
    qa = rng.integers(-63, 64, (M, K)).astype(np.int8)
    qw = rng.integers(-127, 128, (N, K)).astype(np.int8)
    qa[0, :] = 63
    qw[0, :] = -127                                      # extreme magnitudes
    got = oracle.int_block_partials(qa, qw)
    for m in range(M):
        for n in range(N):
            for b in range(K // 32):
                acc = 0
                for kk in range(32 * b, 32 * b + 32):
                    acc += int(qa[m, kk]) * int(qw[n, kk])
                assert got[m, n, b] == acc
    assert got[0, 0, 0] == -63 * 127 * 32


def test_w8a8_linear_within_rounding_bound():
    # With a = s qa + ea (|ea| <= s/2) and w = d qw + ew (|ew| <= d/2),
    # |x.w - y| <= sum_k |s qa| d/2 + s/2 |d qw| + s d / 4.
    rng = np.random.default_rng(2)
    M, N, K = 7, 9, 128
    x = (rng.standard_normal((M, K)) * 3).astype(np.float32)
    x[:, 5] *= 20.0                                      # an outlier channel
    w = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    qw, d = oracle.quantize_weight_blocks(w)
    qa, s = oracle.quantize_rows7(x)
    y = oracle.w8a8_linear(x, qw, d)
    exact = x.astype(np.float64) @ w.astype(np.float64).T
    dk = np.repeat(d.astype(np.float64), 32, axis=1)    # [N, K] scale per element
    sa = s.astype(np.float64)[:, None]
    aq = np.abs(qa.astype(np.float64)) * sa              # [M, K]
    wq = np.abs(qw.astype(np.float64)) * dk              # [N, K]
    bound = (aq @ (dk / 2).T) + (sa / 2) * wq.sum(axis=1)[None, :] + (sa / 4) * dk.sum(axis=1)[None, :]
    assert np.all(np.abs(y - exact) <= bound * (1 + 1e-9) + 1e-12)
    # and it is not trivially exact
    assert np.abs(y - exact).max() > 0


def test_w4a8_model_uses_four_bit_codes():
    from text_embedding_encoder_gb300 import synth
    shape = synth.Shape(n_layers=2, hidden=64, n_heads=1, head_dim=64, intermediate=96, vocab=50)
    w = synth.make_weights(shape, seed=3)
    m = oracle.OracleModel(w, shape, "w4a8")
    for name in ("wqkv", "wo", "wi", "wo_ffn"):
        q, d = m.q[name][1]
        assert np.abs(q).max() == 7
        np.testing.assert_array_equal(q, w8a8.quantize_weight_blocks4(getattr(w, name)[1])[0])
    ids, cu = synth.make_batch([9, 4], shape.vocab, seed=4)
    e4 = oracle.encode_packed(ids, cu, m)
    e8 = oracle.encode_packed(ids, cu, oracle.OracleModel(w, shape, "w8a8"))
    ef = oracle.encode_packed(ids, cu, oracle.OracleModel(w, shape, "fp32"))
    np.testing.assert_allclose(np.linalg.norm(e4, axis=1), 1.0, atol=1e-14)
    # coarser weights: further from the float result than the 8-bit blocks
    assert np.all((e4 * ef).sum(axis=1) < (e8 * ef).sum(axis=1))


def test_w8a8_model_uses_integer_path():
    from text_embedding_encoder_gb300 import synth
    shape = synth.Shape(n_layers=2, hidden=64, n_heads=1, head_dim=64, intermediate=96, vocab=50)
    w = synth.make_weights(shape, seed=3)
    ids, cu = synth.make_batch([9, 4], shape.vocab, seed=4)
    e_int = oracle.encode_packed(ids, cu, oracle.OracleModel(w, shape, "w8a8"))
    e_f = oracle.encode_packed(ids, cu, oracle.OracleModel(w, shape, "fp32"))
    np.testing.assert_allclose(np.linalg.norm(e_int, axis=1), 1.0, atol=1e-14)
    cos = (e_int * e_f).sum(axis=1)
    assert np.all(cos > 0.99) and np.all(cos < 1.0 - 1e-9)
    # the projection goes through quantize -> integer sums -> scales
    m = oracle.OracleModel(w, shape, "w8a8")
    xin = np.random.default_rng(0).standard_normal((3, 64))
    qw, d = w8a8.quantize_weight_blocks(w.wqkv[1])
    qa, s = w8a8.quantize_rows7(xin.astype(np.float32))
    ref = s[:, None].astype(np.float64) * np.einsum("mnb,nb->mn", w8a8.int_block_partials(qa, qw).astype(np.float64),
                                                    d.astype(np.float64))
    np.testing.assert_allclose(m.linear("wqkv", 1, xin), ref, rtol=1e-13, atol=1e-15)


def test_w6a8_model_uses_six_bit_codes():
    from text_embedding_encoder_gb300 import synth
    shape = synth.Shape(n_layers=2, hidden=64, n_heads=1, head_dim=64, intermediate=96, vocab=50)
    w = synth.make_weights(shape, seed=3)
    m = oracle.OracleModel(w, shape, "w6a8")
    for name in ("wqkv", "wo", "wi", "wo_ffn"):
        q, d = m.q[name][1]
        assert np.abs(q).max() == 31
        np.testing.assert_array_equal(q, w8a8.quantize_weight_blocks6(getattr(w, name)[1])[0])
    ids, cu = synth.make_batch([9, 4], shape.vocab, seed=4)
    e6 = oracle.encode_packed(ids, cu, m)
    e4 = oracle.encode_packed(ids, cu, oracle.OracleModel(w, shape, "w4a8"))
    ef = oracle.encode_packed(ids, cu, oracle.OracleModel(w, shape, "fp32"))
    np.testing.assert_allclose(np.linalg.norm(e6, axis=1), 1.0, atol=1e-14)
    # finer weights than the 4-bit blocks: closer to the float result
    assert np.all((e6 * ef).sum(axis=1) > (e4 * ef).sum(axis=1))
