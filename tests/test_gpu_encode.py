"""End-to-end encoder passes through the C ABI on the GPU, against the oracle.

Covers the five workloads (tiny fp32; the 310m shape in bf16 on the
7-text accuracy batch; every text of a full 32768-token sweep batch and of the
2048- and 8192-token sizes; two documents of the 8 x 8192 long-document batch;
the W8A8 path with outlier channels), the
packing invariance the method states (a text's vector does not depend on the
other texts packed with it), edge lengths around the tile and window sizes,
and host-side rejection of malformed input.
"""
import numpy as np
import pytest

import oracle
from text_embedding_encoder_gb300 import binding, synth

torch = pytest.importorskip("torch")
from gpu_util import BF16_COS, assert_embeddings_close, dev, make_encoder, to_np  # noqa: E402

pytestmark = pytest.mark.gpu

W8A8_VS_FP32_COS = 0.99   # W8A8 embeddings against the fp32 path, no outliers


@pytest.fixture(scope="module")
def tiny_weights():
    return synth.make_weights(synth.TINY, seed=0)


@pytest.fixture(scope="module")
def ruri_weights():
    return synth.make_weights(synth.RURI_310M, seed=0)


@pytest.fixture(scope="module")
def ruri_bf16(lib, ruri_weights):
    enc = make_encoder(synth.RURI_310M, "bf16", ruri_weights, max_tokens=65536, max_texts=1024)
    yield enc
    enc.close()


@pytest.fixture(scope="module")
def ruri_oracle_bf16(ruri_weights):
    return oracle.OracleModel(ruri_weights, synth.RURI_310M, "bf16")


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
def test_tiny_config(lib, tiny_weights, dtype):
    ids, cu = synth.make_batch(synth.TINY_LENGTHS, synth.TINY.vocab, seed=0)
    enc = make_encoder(synth.TINY, dtype, tiny_weights, max_tokens=512, max_texts=16)
    got = enc.encode(ids, cu)
    ref = oracle.encode_packed(ids, cu, oracle.OracleModel(tiny_weights, synth.TINY, dtype))
    err = assert_embeddings_close(got, ref, dtype)
    print(f"tiny {dtype}: max abs err {err:.2e}")
    np.testing.assert_allclose(np.linalg.norm(got, axis=1), 1.0, atol=1e-5)
    enc.close()


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
@pytest.mark.parametrize("lengths", [[1], [2], [127, 128, 129], [65, 66, 130], [300], [1, 1, 1]])
def test_tiny_edge_lengths(lib, tiny_weights, dtype, lengths):
    ids, cu = synth.make_batch(lengths, synth.TINY.vocab, seed=sum(lengths))
    enc = make_encoder(synth.TINY, dtype, tiny_weights, max_tokens=sum(lengths), max_texts=len(lengths))
    got = enc.encode(ids, cu)
    ref = oracle.encode_packed(ids, cu, oracle.OracleModel(tiny_weights, synth.TINY, dtype))
    assert_embeddings_close(got, ref, dtype)
    enc.close()


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
def test_packing_invariance(lib, tiny_weights, dtype):
    lengths = [37, 150, 8, 64, 129]
    ids, cu = synth.make_batch(lengths, synth.TINY.vocab, seed=9)
    enc = make_encoder(synth.TINY, dtype, tiny_weights, max_tokens=512, max_texts=16)
    packed = enc.encode(ids, cu)
    alone = np.stack([enc.encode(ids[a:b], np.array([0, b - a], np.int32)) [0] for a, b in zip(cu[:-1], cu[1:])])
    # reversed packing order
    order = list(range(len(lengths)))[::-1]
    ids_r = np.concatenate([ids[cu[j]:cu[j + 1]] for j in order])
    cu_r = np.concatenate([[0], np.cumsum([lengths[j] for j in order])]).astype(np.int32)
    rev = enc.encode(ids_r, cu_r)[::-1]
    # fp32: bit-identical (the SIMT attention visits each row's keys in the same
    # order however the texts are packed).  bf16: the window layers tile the
    # packed sequence itself, so which 128-key tile (and which softmax warp's
    # reference maximum) a key falls in depends on the neighbouring texts; the
    # bf16 rounding of P then differs, by about 2e-4 on these vectors, well
    # inside the 3e-3 bar against the oracle
    tol = 0.0 if dtype == "fp32" else 1e-3
    np.testing.assert_allclose(packed, alone, atol=tol, rtol=0)
    np.testing.assert_allclose(packed, rev, atol=tol, rtol=0)
    sim = packed @ packed.T
    np.testing.assert_allclose(np.diag(sim), 1.0, atol=2e-6)
    np.testing.assert_allclose(sim, sim.T, atol=1e-6)
    enc.close()


def test_ruri_accuracy_batch_bf16(ruri_bf16, ruri_oracle_bf16):
    ids, cu = synth.make_batch(synth.ACCURACY_LENGTHS, synth.RURI_310M.vocab, seed=0)
    got = ruri_bf16.encode(ids, cu)
    ref = oracle.encode_packed(ids, cu, ruri_oracle_bf16)
    err = assert_embeddings_close(got, ref, "bf16")
    cos = np.sum(got * ref, axis=1)
    print(f"310m bf16 accuracy batch: max abs {err:.2e}, min cos {cos.min():.6f}")


def test_ruri_sweep_32k_every_text(ruri_bf16, ruri_oracle_bf16):
    """Full 32768-token sweep batch in the bench's launch configuration
    (device buffers, tee_encode_device); every text checked by the oracle.
    The attention work list is sorted longest first and spread over persistent
    CTAs, so a scheduling mistake could hit any text."""
    ids, cu = synth.sweep_batch(32768, 0, synth.RURI_310M.vocab)
    n = len(cu) - 1
    out = torch.empty(n, synth.RURI_310M.hidden, device="cuda")
    ruri_bf16.encode_device(dev(ids), dev(cu), cu, out, 0)
    torch.cuda.synchronize()
    got = to_np(out)
    ref = oracle.encode_packed(ids, cu, ruri_oracle_bf16)
    err = assert_embeddings_close(got, ref, "bf16")
    cos = np.sum(got * ref, axis=1)
    print(f"32k sweep batch 0, {n} texts: max abs {err:.2e}, min cos {cos.min():.6f}")
    np.testing.assert_allclose(np.linalg.norm(got, axis=1), 1.0, atol=1e-5)


@pytest.mark.parametrize("budget,batch", [(2048, 3), (8192, 7)])
def test_ruri_small_sweeps_every_text(ruri_bf16, ruri_oracle_bf16, budget, batch):
    """The 2048- and 8192-token sweep sizes take other GEMM tilings (single
    CTAs and 192-column CTA pairs on the long-K projection) and fewer
    attention units than 32768; every text against the oracle."""
    ids, cu = synth.sweep_batch(budget, batch, synth.RURI_310M.vocab)
    out = torch.empty(len(cu) - 1, synth.RURI_310M.hidden, device="cuda")
    ruri_bf16.encode_device(dev(ids), dev(cu), cu, out, 0)
    torch.cuda.synchronize()
    got = to_np(out)
    ref = oracle.encode_packed(ids, cu, ruri_oracle_bf16)
    assert_embeddings_close(got, ref, "bf16")
    np.testing.assert_allclose(np.linalg.norm(got, axis=1), 1.0, atol=1e-5)


def test_ruri_long_docs_two_texts(ruri_bf16, ruri_oracle_bf16):
    """8 x 8192 tokens: the first and a middle document against the oracle
    (each alone is a full 8192-token global-attention text)."""
    ids, cu = synth.make_batch(synth.LONG_DOC_LENGTHS, synth.RURI_310M.vocab, seed=0)
    got = ruri_bf16.encode(ids, cu)
    sample = [0, 5]
    ref = oracle.encode_packed(ids, cu, ruri_oracle_bf16, texts=sample)
    assert_embeddings_close(got[sample], ref[sample], "bf16")
    np.testing.assert_allclose(np.linalg.norm(got, axis=1), 1.0, atol=1e-5)


def test_two_contexts_interleaved_on_one_device(lib, tiny_weights):
    """Two contexts (different shapes and arithmetic) used alternately in one
    process: each entry point makes its own context's device current and puts
    the caller's back, and the launchers keep their per-device state apart."""
    odd = synth.Shape(n_layers=2, hidden=384, n_heads=6, head_dim=64, intermediate=640, vocab=1000)
    w_odd = synth.make_weights(odd, seed=4)
    a = make_encoder(synth.TINY, "bf16", tiny_weights, max_tokens=512, max_texts=16)
    b = make_encoder(odd, "bf16", w_odd, max_tokens=512, max_texts=16)
    c = make_encoder(synth.TINY, "fp32", tiny_weights, max_tokens=512, max_texts=16)
    ids_t, cu_t = synth.make_batch([37, 150, 8, 64], synth.TINY.vocab, seed=2)
    ids_o, cu_o = synth.make_batch([129, 3, 200], odd.vocab, seed=3)
    ref_a = oracle.encode_packed(ids_t, cu_t, oracle.OracleModel(tiny_weights, synth.TINY, "bf16"))
    ref_b = oracle.encode_packed(ids_o, cu_o, oracle.OracleModel(w_odd, odd, "bf16"))
    ref_c = oracle.encode_packed(ids_t, cu_t, oracle.OracleModel(tiny_weights, synth.TINY, "fp32"))
    before = torch.cuda.current_device()
    for _ in range(3):
        assert_embeddings_close(a.encode(ids_t, cu_t), ref_a, "bf16")
        assert_embeddings_close(b.encode(ids_o, cu_o), ref_b, "bf16")
        assert_embeddings_close(c.encode(ids_t, cu_t), ref_c, "fp32")
    assert torch.cuda.current_device() == before
    for e in (a, b, c):
        e.close()


@pytest.mark.parametrize("outliers", [False, True])
def test_tiny_w8a8(lib, outliers):
    shape = synth.TINY
    w = synth.make_weights(shape, seed=0, outliers=outliers)
    ids, cu = synth.make_batch(synth.TINY_LENGTHS, shape.vocab, seed=0)
    enc = make_encoder(shape, "w8a8", w, max_tokens=512, max_texts=16)
    got = enc.encode(ids, cu)
    enc.close()
    ref = oracle.encode_packed(ids, cu, oracle.OracleModel(w, shape, "w8a8"))
    cos = np.sum(got * ref, axis=1)
    print(f"tiny w8a8 outliers={outliers}: min cos vs W8A8 oracle {cos.min():.7f}")
    assert cos.min() >= 0.9995


@pytest.mark.parametrize("outliers", [False, True])
def test_ruri_w8a8(lib, outliers):
    """The 310m shape through the integer path.  Without outliers the GPU must
    agree with the W8A8 oracle like the bf16 path does.  With the 20x outlier
    channels the procedure is chaotic: one flipped 7-bit code (the GPU decides
    codes from fp32 activations, the oracle from fp64 ones rounded to fp32)
    changes a whole coarse quantisation step, and 25 layers amplify it -- the
    oracle itself moves to cosine 0.973 on one of these texts when its
    embedding table is perturbed by 1e-7 relative.  There the bar is 0.95, and
    the int8 codes and int32 block sums are checked bit-exactly by the
    step tests."""
    shape = synth.RURI_310M
    w = synth.make_weights(shape, seed=0, outliers=outliers)
    ids, cu = synth.make_batch(synth.ACCURACY_LENGTHS, shape.vocab, seed=0)
    enc = make_encoder(shape, "w8a8", w, max_tokens=2048, max_texts=16)
    got = enc.encode(ids, cu)
    enc.close()
    ref_int = oracle.encode_packed(ids, cu, oracle.OracleModel(w, shape, "w8a8"))
    ref_f = oracle.encode_packed(ids, cu, oracle.OracleModel(w, shape, "fp32"))
    cos_int = np.sum(got * ref_int, axis=1)
    cos_f = np.sum(got * ref_f, axis=1)
    cos_oracles = np.sum(ref_int * ref_f, axis=1)
    print(f"310m w8a8 outliers={outliers}: min cos vs W8A8 oracle {cos_int.min():.6f}; vs fp32 oracle "
          f"{cos_f.min():.6f} (W8A8 oracle vs fp32 oracle: {cos_oracles.min():.6f})")
    assert cos_int.min() >= (0.95 if outliers else BF16_COS)
    np.testing.assert_allclose(np.linalg.norm(got, axis=1), 1.0, atol=1e-5)
    if not outliers:
        # against the fp32 path: the page's -q8 stays at cosine >= 0.9912 of the
        # unquantised model on its trained weights; the bar here is 0.99
        assert cos_f.min() >= W8A8_VS_FP32_COS, cos_f.min()
    else:
        # with 20x outlier channels the outliers set every row's 7-bit scale, so
        # the other channels keep a few levels each and the W8A8 procedure itself
        # is far from fp32 (the W8A8 oracle is at about 0.76 of the fp32 oracle);
        # the GPU must not be further from fp32 than that procedure is
        assert cos_f.min() >= cos_oracles.min() - 0.05, (cos_f.min(), cos_oracles.min())


def test_host_validation_and_recovery(lib, tiny_weights):
    enc = binding.Encoder(synth.TINY, "fp32", max_tokens=64, max_texts=4)
    ids, cu = synth.make_batch([5, 7], synth.TINY.vocab, seed=1)
    with pytest.raises(binding.TeeError) as e:
        enc.encode(ids, cu)
    assert e.value.code == binding.TEE_ENOTLOADED
    enc.load_weights(tiny_weights)
    bad = [
        (ids, np.array([1, 5, 12], np.int32), binding.TEE_EINVAL),          # cu[0] != 0
        (ids, np.array([0, 5, 5], np.int32), binding.TEE_EINVAL),           # empty text
        (ids, np.array([0, 7, 5], np.int32), binding.TEE_EINVAL),           # decreasing
        (np.zeros(65, np.int32), np.array([0, 65], np.int32), binding.TEE_ETOOLONG),
        (np.array([1, 5000, 2], np.int32), np.array([0, 3], np.int32), binding.TEE_EINVAL),   # id >= vocab
        (np.array([1, -3, 2], np.int32), np.array([0, 3], np.int32), binding.TEE_EINVAL),
        (ids, np.array([0], np.int32), binding.TEE_EINVAL),                 # no texts
        (np.zeros(10, np.int32), np.arange(6, dtype=np.int32) * 2, binding.TEE_ETOOLONG),   # 5 texts > 4
    ]
    for bi, bc, code in bad:
        with pytest.raises(binding.TeeError) as e:
            enc.encode(bi, bc)
        assert e.value.code == code, (bc, e.value)
    good = enc.encode(ids, cu)   # still usable
    ref = oracle.encode_packed(ids, cu, oracle.OracleModel(tiny_weights, synth.TINY, "fp32"))
    assert_embeddings_close(good, ref, "fp32")
    # device path: an out-of-range id is reported through the status word
    out = torch.empty(1, synth.TINY.hidden, device="cuda")
    enc.encode_device(dev(np.array([1, 99999, 2], np.int32)), dev(np.array([0, 3], np.int32)),
                      np.array([0, 3], np.int32), out, 0)
    assert enc.device_status() == binding.TEE_EINVAL
    assert enc.device_status() == 0
    enc.close()


def test_bounded_wait_expiry_is_reported(lib, tiny_weights):
    """A device wait that runs out (on a barrier nothing completes, ~1 ms limit)
    is reported as TEE_ETIMEOUT through the status word, once, and the context
    keeps working afterwards."""
    enc = make_encoder(synth.TINY, "bf16", tiny_weights, max_tokens=512, max_texts=16)
    assert enc.device_status() == binding.TEE_OK
    enc.check(lib.tee_selftest_wait_timeout(enc.ctx, 2_000_000, None))
    assert enc.device_status() == binding.TEE_ETIMEOUT
    assert enc.device_status() == binding.TEE_OK
    ids, cu = synth.make_batch(synth.TINY_LENGTHS, synth.TINY.vocab, seed=0)
    got = enc.encode(ids, cu)
    ref = oracle.encode_packed(ids, cu, oracle.OracleModel(tiny_weights, synth.TINY, "bf16"))
    assert_embeddings_close(got, ref, "bf16")
    enc.close()
